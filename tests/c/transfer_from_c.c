/* A transfer through libkvx's C ABI from a plain C99 program (no Python, no C++): two
 * per-plane token pools in device memory, a request of distinct slots, the move checked row by
 * row against its definition (row(dst, p, d[i]) = row(src, p, s[i]), every other destination
 * row untouched), then a request with one slot past the end, which must move nothing.
 * Exit status 0 and "ok" on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvx.h"

#define CHECK_CUDA(x)                                                        \
  do {                                                                       \
    cudaError_t e_ = (x);                                                    \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
      return 1;                                                              \
    }                                                                        \
  } while (0)

#define CHECK_KVX(x)                                                         \
  do {                                                                       \
    kvx_status s_ = (x);                                                     \
    if (s_ != KVX_OK) {                                                      \
      fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, kvx_status_str(s_)); \
      return 1;                                                              \
    }                                                                        \
  } while (0)

enum { L = 3, H = 2, D = 64, NUM = 1000, N = 300 };

static unsigned char pattern(int64_t plane, int64_t slot, int64_t byte) {
  return (unsigned char)((plane * 131 + slot * 7 + byte * 3 + 1) & 0xFF);
}

int main(void) {
  const int64_t R = (int64_t)H * D * 2, P = 2 * L, pool = P * NUM * R;
  unsigned char *h_src = (unsigned char *)malloc((size_t)pool);
  unsigned char *h_dst = (unsigned char *)malloc((size_t)pool);
  int32_t s[N], d[N];
  int64_t p, j, i, b;
  void *d_src, *d_dst, *d_ws;
  int32_t *d_s, *d_d, *d_status, status = -1;
  kvx_layout_desc desc;
  kvx_layout_t src_l, dst_l;
  size_t ws_bytes;
  if (!h_src || !h_dst) return 1;
  for (p = 0; p < P; ++p)
    for (j = 0; j < NUM; ++j)
      for (b = 0; b < R; ++b) h_src[(p * NUM + j) * R + b] = pattern(p, j, b);
  for (i = 0; i < N; ++i) {
    s[i] = (int32_t)((7 * i + 3) % NUM); /* distinct: 7 and 1000 are coprime */
    d[i] = (int32_t)((13 * i + 5) % NUM);
  }
  CHECK_CUDA(cudaMalloc(&d_src, (size_t)pool));
  CHECK_CUDA(cudaMalloc(&d_dst, (size_t)pool));
  CHECK_CUDA(cudaMalloc((void **)&d_s, sizeof s));
  CHECK_CUDA(cudaMalloc((void **)&d_d, sizeof d));
  CHECK_CUDA(cudaMalloc((void **)&d_status, 16));
  CHECK_CUDA(cudaMemcpy(d_src, h_src, (size_t)pool, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemset(d_dst, 0xFF, (size_t)pool));
  CHECK_CUDA(cudaMemcpy(d_s, s, sizeof s, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(d_d, d, sizeof d, cudaMemcpyHostToDevice));

  memset(&desc, 0, sizeof desc);
  desc.num_layers = L;
  desc.kv_heads = H;
  desc.head_dim = D;
  desc.dtype = KVX_BF16;
  desc.kind = KVX_NHD;
  desc.num_slots = NUM;
  desc.plane_stride = NUM * R;
  desc.base = d_src;
  CHECK_KVX(kvx_layout_create(&desc, &src_l));
  desc.base = d_dst;
  CHECK_KVX(kvx_layout_create(&desc, &dst_l));
  if (kvx_layout_row_bytes(src_l) != R || kvx_layout_num_planes(src_l) != P) return 1;
  ws_bytes = kvx_workspace_size(N, 0);
  if (ws_bytes == 0) return 1;
  CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));

  CHECK_KVX(kvx_transfer(src_l, d_s, dst_l, d_d, N, d_ws, ws_bytes, d_status, KVX_DEFAULTS, NULL));
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(&status, d_status, sizeof status, cudaMemcpyDeviceToHost));
  if (status != KVX_OK) {
    fprintf(stderr, "status %s\n", kvx_status_str((kvx_status)status));
    return 1;
  }
  CHECK_CUDA(cudaMemcpy(h_dst, d_dst, (size_t)pool, cudaMemcpyDeviceToHost));
  {
    int32_t *src_of = (int32_t *)malloc(sizeof(int32_t) * NUM); /* -1: slot not written */
    if (!src_of) return 1;
    for (j = 0; j < NUM; ++j) src_of[j] = -1;
    for (i = 0; i < N; ++i) src_of[d[i]] = s[i];
    for (p = 0; p < P; ++p)
      for (j = 0; j < NUM; ++j)
        for (b = 0; b < R; ++b) {
          const unsigned char got = h_dst[(p * NUM + j) * R + b];
          const unsigned char want = src_of[j] < 0 ? 0xFF : pattern(p, src_of[j], b);
          if (got != want) {
            fprintf(stderr, "plane %lld slot %lld byte %lld: %u, want %u\n", (long long)p,
                    (long long)j, (long long)b, got, want);
            return 1;
          }
        }
    free(src_of);
  }

  /* one source slot past the end: refused on the device, nothing moved */
  s[N / 2] = NUM;
  CHECK_CUDA(cudaMemcpy(d_s, s, sizeof s, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemset(d_dst, 0xFF, (size_t)pool));
  CHECK_KVX(kvx_transfer(src_l, d_s, dst_l, d_d, N, d_ws, ws_bytes, d_status, 0u, NULL));
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(&status, d_status, sizeof status, cudaMemcpyDeviceToHost));
  if (status != KVX_ERR_OUT_OF_RANGE) return 1;
  CHECK_CUDA(cudaMemcpy(h_dst, d_dst, (size_t)pool, cudaMemcpyDeviceToHost));
  for (b = 0; b < pool; ++b)
    if (h_dst[b] != 0xFF) return 1;

  kvx_layout_destroy(src_l);
  kvx_layout_destroy(dst_l);
  cudaFree(d_src);
  cudaFree(d_dst);
  cudaFree(d_s);
  cudaFree(d_d);
  cudaFree(d_status);
  cudaFree(d_ws);
  free(h_src);
  free(h_dst);
  printf("ok\n");
  return 0;
}

/* A plain C client of libringattn.so, with no Python or PyTorch involved: it reads
 * q, k, v (raw bf16, [B, N, H, d] and [B, N, G, d]) from a directory, allocates device
 * buffers with the CUDA runtime, runs ring_attn_fwd on them and writes o (raw bf16)
 * and lse (raw fp32, [B, H, N]) back. It also checks that a malformed problem is
 * refused before any launch.
 *
 *   c_client DIR B N H G d P causal layout
 *
 * Exit status: 0 on success, 1 on an I/O or CUDA runtime error, 2 when the library
 * returns an unexpected status, 3 when the device status word is not clean. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ringattn.h"

static int read_file(const char* dir, const char* name, void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (f == NULL) return 1;
  const size_t got = fread(buf, 1, bytes, f);
  fclose(f);
  return got == bytes ? 0 : 1;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (f == NULL) return 1;
  const size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : 1;
}

int main(int argc, char** argv) {
  if (argc != 10) {
    fprintf(stderr, "usage: %s DIR B N H G d P causal layout\n", argv[0]);
    return 1;
  }
  const char* dir = argv[1];
  ra_problem p;
  p.batch = atoi(argv[2]);
  p.seqlen = atoi(argv[3]);
  p.heads = atoi(argv[4]);
  p.kv_heads = atoi(argv[5]);
  p.head_dim = atoi(argv[6]);
  p.P = atoi(argv[7]);
  p.causal = atoi(argv[8]);
  p.layout = atoi(argv[9]);
  p.scale = 0.f;
  p.o_dtype = RA_DTYPE_BF16;
  const size_t tok = (size_t)p.batch * (size_t)p.seqlen;
  const size_t bq = tok * (size_t)p.heads * (size_t)p.head_dim * 2;
  const size_t bkv = tok * (size_t)p.kv_heads * (size_t)p.head_dim * 2;
  const size_t bl = tok * (size_t)p.heads * sizeof(float);

  void* hq = malloc(bq);
  void* hk = malloc(bkv);
  void* hv = malloc(bkv);
  void* ho = malloc(bq);
  void* hl = malloc(bl);
  if (!hq || !hk || !hv || !ho || !hl) return 1;
  if (read_file(dir, "q.bin", hq, bq) || read_file(dir, "k.bin", hk, bkv) ||
      read_file(dir, "v.bin", hv, bkv))
    return 1;

  void *dq = NULL, *dk = NULL, *dv = NULL, *d_o = NULL, *dl = NULL;
  if (cudaMalloc(&dq, bq) != cudaSuccess || cudaMalloc(&dk, bkv) != cudaSuccess ||
      cudaMalloc(&dv, bkv) != cudaSuccess || cudaMalloc(&d_o, bq) != cudaSuccess ||
      cudaMalloc(&dl, bl) != cudaSuccess)
    return 1;
  if (cudaMemcpy(dq, hq, bq, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(dk, hk, bkv, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(dv, hv, bkv, cudaMemcpyHostToDevice) != cudaSuccess)
    return 1;

  /* A malformed problem (H not a multiple of G) is refused before any launch. */
  ra_problem bad = p;
  bad.kv_heads = p.heads + 1;
  if (ring_attn_fwd(&bad, dq, dk, dv, d_o, (float*)dl, NULL) != RA_ERR_INVALID_ARG) return 2;

  const ra_status st = ring_attn_fwd(&p, dq, dk, dv, d_o, (float*)dl, NULL);
  if (st != RA_OK) {
    fprintf(stderr, "ring_attn_fwd: %s\n", ra_status_str(st));
    return 2;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  int32_t code = -1;
  if (ring_attn_last_error(&code) != RA_OK || code != 0) return 3;

  if (cudaMemcpy(ho, d_o, bq, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(hl, dl, bl, cudaMemcpyDeviceToHost) != cudaSuccess)
    return 1;
  if (write_file(dir, "o.bin", ho, bq) || write_file(dir, "lse.bin", hl, bl)) return 1;
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(d_o);
  cudaFree(dl);
  free(hq);
  free(hk);
  free(hv);
  free(ho);
  free(hl);
  printf("ok %s\n", ra_status_str(st));
  return 0;
}

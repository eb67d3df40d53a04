/* A plain C11 user of include/taco.h and libtaco.so: compress one bf16
 * tensor and decompress-reduce it through the C ABI, from host buffers
 * copied in and out with cudaMemcpy, then check that bad arguments are
 * rejected with their status and write nothing.
 *
 * usage: c_roundtrip <x.bin> <N> <h> <block> <out prefix>
 *   x.bin      N*h bf16 values (raw little-endian bits)
 *   writes     <prefix>.codes (N*h bytes), <prefix>.scales (N*h/block
 *              (alpha, s) fp32 pairs), <prefix>.out (N*h bf16)
 * Exit status 0 on success; a message on stderr otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "taco.h"

#define CHECK_CUDA(call)                                                     \
  do {                                                                       \
    cudaError_t e_ = (call);                                                 \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
      return 2;                                                              \
    }                                                                        \
  } while (0)

#define EXPECT(call, status)                                                 \
  do {                                                                       \
    taco_status s_ = (call);                                                 \
    if (s_ != (status)) {                                                    \
      fprintf(stderr, "%s returned %d (%s), expected %d\n", #call, (int)s_,  \
              taco_status_string(s_), (int)(status));                        \
      return 3;                                                              \
    }                                                                        \
  } while (0)

static int write_file(const char* prefix, const char* ext, const void* p, size_t n) {
  char path[4096];
  snprintf(path, sizeof path, "%s.%s", prefix, ext);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(p, 1, n, f) != n) return 1;
  return fclose(f) != 0;
}

int main(int argc, char** argv) {
  if (argc != 6) {
    fprintf(stderr, "usage: %s x.bin N h block prefix\n", argv[0]);
    return 1;
  }
  const int64_t N = atoll(argv[2]), h = atoll(argv[3]);
  const int block = atoi(argv[4]);
  const size_t elems = (size_t)(N * h);
  const size_t shard = taco_shard_bytes(N, h, block);
  const size_t scales_off = taco_shard_scales_offset(N, h, block);
  const size_t ws_bytes = taco_workspace_bytes(1);
  if (shard == 0 || ws_bytes == 0) return 1;

  uint16_t* x = malloc(elems * 2);
  uint8_t* bundle = malloc(shard);
  uint16_t* out = malloc(elems * 2);
  uint16_t* again = malloc(elems * 2);
  FILE* f = fopen(argv[1], "rb");
  if (!x || !bundle || !out || !again || !f || fread(x, 2, elems, f) != elems) return 1;
  fclose(f);

  void *dx, *dbundle, *dheader, *dws, *dout;
  CHECK_CUDA(cudaMalloc(&dx, elems * 2));
  CHECK_CUDA(cudaMalloc(&dbundle, shard));
  CHECK_CUDA(cudaMalloc(&dheader, sizeof(taco_header)));
  CHECK_CUDA(cudaMalloc(&dws, ws_bytes));
  CHECK_CUDA(cudaMalloc(&dout, elems * 2));
  CHECK_CUDA(cudaMemset(dws, 0, ws_bytes));   /* zero before its first use */
  CHECK_CUDA(cudaMemcpy(dx, x, elems * 2, cudaMemcpyHostToDevice));

  EXPECT(taco_compress(dx, N, h, block, 4096.0f, TACO_VARIANT_DUAL, dbundle, dheader, dws,
                       ws_bytes, NULL), TACO_OK);
  EXPECT(taco_decompress_reduce(dbundle, 1, N, h, block, dout, NULL), TACO_OK);
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(bundle, dbundle, shard, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(out, dout, elems * 2, cudaMemcpyDeviceToHost));
  taco_header hdr;
  CHECK_CUDA(cudaMemcpy(&hdr, dheader, sizeof hdr, cudaMemcpyDeviceToHost));
  if (hdr.N != N || hdr.h != h || hdr.block != block || hdr.q_max != TACO_Q_MAX) {
    fprintf(stderr, "header fields differ\n");
    return 4;
  }

  /* Every bad argument is rejected before anything is launched: the output
   * buffers keep what the good calls wrote. */
  EXPECT(taco_compress(dx, N, h, 100, 4096.0f, 0, dbundle, dheader, dws, ws_bytes, NULL), TACO_ERR_BLOCK);
  EXPECT(taco_compress(dx, N, h + 1, block, 4096.0f, 0, dbundle, dheader, dws, ws_bytes, NULL), TACO_ERR_SHAPE);
  EXPECT(taco_compress((char*)dx + 2, N, h, block, 4096.0f, 0, dbundle, dheader, dws, ws_bytes, NULL),
         TACO_ERR_ALIGN);
  EXPECT(taco_compress(dx, N, h, block, -1.0f, 0, dbundle, dheader, dws, ws_bytes, NULL), TACO_ERR_ARG);
  EXPECT(taco_compress(dx, N, h, block, 4096.0f, 7, dbundle, dheader, dws, ws_bytes, NULL), TACO_ERR_ARG);
  EXPECT(taco_compress(dx, N, h, block, 4096.0f, 0, dbundle, dheader, dws, 0, NULL), TACO_ERR_WORKSPACE);
  EXPECT(taco_compress(dx, N, h, block, 4096.0f, 0, NULL, dheader, dws, ws_bytes, NULL), TACO_ERR_NULL);
  EXPECT(taco_decompress_reduce(NULL, 1, N, h, block, dout, NULL), TACO_ERR_NULL);
  EXPECT(taco_decompress_reduce(dbundle, 0, N, h, block, dout, NULL), TACO_ERR_ARG);
  EXPECT(taco_decompress_reduce(dbundle, TACO_MAX_SHARDS + 1, N, h, block, dout, NULL), TACO_ERR_ARG);
  EXPECT(taco_decompress_reduce(dbundle, 1, N, h, block, (char*)dout + 8, NULL), TACO_ERR_ALIGN);
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(again, dout, elems * 2, cudaMemcpyDeviceToHost));
  if (memcmp(again, out, elems * 2) != 0) {
    fprintf(stderr, "a rejected call changed the output\n");
    return 5;
  }

  if (write_file(argv[5], "codes", bundle, elems) ||
      write_file(argv[5], "scales", bundle + scales_off, elems / (size_t)block * 8) ||
      write_file(argv[5], "out", out, elems * 2))
    return 1;
  cudaFree(dx);
  cudaFree(dbundle);
  cudaFree(dheader);
  cudaFree(dws);
  cudaFree(dout);
  free(x);
  free(bundle);
  free(out);
  free(again);
  printf("ok\n");
  return 0;
}

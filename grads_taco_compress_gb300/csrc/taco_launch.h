// Internal launch interface between the C ABI (taco_abi.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "taco.h"

namespace taco {

constexpr int kCompressThreads = 256;
constexpr int kDecompressThreads = 256;

// Workspace of compress: per shard one arrival counter (16 bytes) followed by
// one (max s, count) pair per CTA of the shard's grid row.
constexpr int kMaxCtasPerShard = 2048;
constexpr size_t kWorkspaceShardStride = 16 + 8 * static_cast<size_t>(kMaxCtasPerShard);

struct CompressArgs {
  const uint16_t* x;        // [P][N][h] bf16
  int64_t shard_elems;      // N * h
  int64_t nblocks;          // N * h / block
  uint8_t* bundle;          // P shards
  size_t shard_bytes;
  size_t alpha_off;
  size_t s_off;
  taco_header* headers;     // [P]
  uint8_t* workspace;
  int64_t N;
  int64_t h;
  float target_energy;
  float sqrt_nE;            // fp32(sqrt(block * E*))
  float inv_sqrt_n;         // fp32(1 / sqrt(block))
};

struct DecompressArgs {
  const uint8_t* shard[TACO_MAX_SHARDS];   // shard p base
  size_t alpha_off;
  size_t s_off;
  int P;
  int64_t nblocks;
  uint16_t* out;            // [N][h] bf16
  float inv_sqrt_n;
};

int compress_tile_blocks(int block);
const void* compress_kernel_ptr(int block, int variant);
cudaError_t launch_compress(const CompressArgs& a, int block, int variant, int grid_x, int P,
                            cudaStream_t stream);

int decompress_tile_blocks(int block);
const void* decompress_kernel_ptr(int block);
cudaError_t launch_decompress(const DecompressArgs& a, int block, int grid, cudaStream_t stream);

}  // namespace taco

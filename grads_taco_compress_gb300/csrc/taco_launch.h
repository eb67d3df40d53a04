// Internal launch interface between the C ABI (taco_abi.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "taco.h"

namespace taco {

// CUDA-core compress: 16 warps in one CTA per SM (192 KB of stages); two CTAs
// of 8 warps measured slower on the large tensors (gpt3-act 0.900 -> 0.943 of
// the measured peak with one CTA) and 1.4% faster on gpt2.
constexpr int kCompressThreads = 512;
constexpr int kCompressMinBlocks = 1;
constexpr int kCompressStages = 3;        // warp tiles (4 KB each) in flight per warp
// Decompress-reduce: 16 warps in one CTA per SM (213.5 KB of stages and
// output buffers). Two CTAs of 8 warps per SM measured slower: the warps of
// the CTA resident first were favoured and the other CTA finished alone.
constexpr int kDecompressThreads = 512;
constexpr int kDecompressMinBlocks = 1;
constexpr int kDecompressStages = 4;      // (tile, shard) stages in flight per warp
constexpr int64_t kClaimRounds = 3;      // decompress-reduce: claimed tiles from this many rounds per warp
constexpr int kVariants = 3;              // DUAL, ABSMAX, STATIC
// Tensor-core compress: a producer warp, an MMA warp, groups of 4 epilogue
// warps (one accumulator of `block` TMEM columns per group) and a tile
// scheduler warp.
constexpr int compress_mma_groups(int) { return 2; }
constexpr int compress_mma_threads(int block) { return 64 + 128 * compress_mma_groups(block) + 32; }
// Largest blocks per shard of the tensor-core compress (32-bit TMA coordinates).
constexpr int64_t kMmaMaxBlocks = (int64_t{1} << 31) - 256;

// Largest grid row (CTAs per shard) of any launch.
constexpr int kMaxCtasPerShard = 2048;
// Workspace of one shard: 16 bytes, zero between calls. Each kernel lays out
// its header counters there (taco_device.cuh, compress_mma.cu); the first
// shard's slot also holds the tensor-core compress's launch-wide tile pool.
constexpr size_t kWorkspaceShardStride = 16;

struct CompressArgs {
  const uint16_t* x;        // [P][N][h] bf16
  int64_t shard_elems;      // N * h
  int64_t nblocks;          // N * h / block
  uint8_t* bundle;          // P shards
  size_t shard_bytes;
  size_t scales_off;        // (alpha, s) float2 per block
  taco_header* headers;     // [P]
  uint8_t* workspace;
  int64_t N;
  int64_t h;
  float target_energy;
  float sqrt_nE;            // fp32(sqrt(block * E*))
  float inv_sqrt_n;         // fp32(1 / sqrt(block))
  float s_static;           // fp32(sqrt(block * E*) / 448), STATIC variant
  float n_sqrtE;            // fp32(block * sqrt(E*)), tensor-core compress
  float q_max;              // largest code magnitude written to the headers (448 or 127)
};

struct DecompressArgs {
  const uint8_t* shard[TACO_MAX_SHARDS];   // shard p base
  size_t scales_off;
  int P;
  int64_t nblocks;
  uint16_t* out;            // [N][h] bf16 (reduce-recompress: may be null)
  float inv_sqrt_n;
  // reduce-recompress only: the compressed sum and its header
  uint8_t* rc_shard;        // codes | (alpha, s) pairs, same layout as the inputs
  taco_header* rc_header;
  uint8_t* workspace;       // one header workspace per reduced shard
  size_t rc_stride;         // bytes between the reduced shards of a batched launch
                            // (gridDim.y reductions of P shards each)
  int64_t N;
  int64_t h;
  float target_energy;
  float sqrt_E;             // fp32(sqrt(E*))
  float sqrt_n;             // fp32(sqrt(block))
  float s_static;           // fp32(sqrt(block * E*) / 448), STATIC variant
};

// The argument checks of the compress entry points, without any CUDA call:
// TACO_OK, or the status such a call returns before it enqueues anything.
taco_status check_compress_args(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                                float target_energy, int variant, const void* bundle_out,
                                const taco_header* headers_out, const void* workspace,
                                size_t workspace_bytes);

size_t compress_smem_bytes();
const void* compress_kernel_ptr(int block, int variant);
cudaError_t launch_compress(const CompressArgs& a, int block, int variant, int grid_x, int P,
                            cudaStream_t stream);
cudaError_t compress_fault(unsigned int* bits, bool clear);

size_t compress_mma_smem_bytes(int block);
// fmt: 0 = FP8 E4M3 codes, 1 = INT8 fallback codes
const void* compress_mma_kernel_ptr(int block, int variant, int fmt);
cudaError_t launch_compress_mma(const CompressArgs& a, int block, int variant, int fmt, int grid_x,
                                int P, cudaStream_t stream);
cudaError_t compress_mma_fault(unsigned int* bits, bool clear);

size_t decompress_smem_bytes();
const void* decompress_kernel_ptr(int block, int fmt, bool claim);
// Producer-warp kernels (decompress_pw.cu): mode 0 decompress-reduce, mode 1
// reduce-recompress (gridDim.y = batch reductions), any block and format.
size_t decompress_pw_smem_bytes(int block);
int64_t decompress_pw_tile_blocks(int block);
const void* decompress_pw_kernel_ptr(int mode, int block, int variant, int fmt);
cudaError_t launch_decompress_pw(const DecompressArgs& a, int mode, int block, int variant, int fmt,
                                 int grid, int batch, cudaStream_t stream);
cudaError_t decompress_pw_fault(unsigned int* bits, bool clear);
// Whether a launch of this mode (0 decompress-reduce, 1 reduce-recompress),
// block size and code format runs the producer-warp kernel. Measured against
// the per-warp-copy kernel (decompress_reduce.cu), back-to-back launches on
// GB300: n = 64 is faster in every mode and format (gpt2-1.5b-act: E4M3
// decompress-reduce equal at 15.57 us, INT8 17.11 -> 15.82 us,
// reduce-recompress 17.01 -> 15.22 us E4M3 and 17.92 -> 15.90 us INT8); at
// n = 128 and 256 the per-warp copies with claimed tiles stay ahead by 1-10%
// (gpt3-6.7b-act decompress-reduce 56.7 us against 59.5 us).
inline bool decompress_uses_pw(int mode, int block, int fmt) {
  (void)mode;
  (void)fmt;
  return block == 64;
}
// The fewest blocks a CTA of the producer-warp kernel is given (two of its
// consumer warps' worth), so that small tensors still spread over many SMs.
constexpr int64_t kPwMinBlocksPerCta = 64;
cudaError_t launch_decompress(const DecompressArgs& a, int block, int fmt, int grid,
                              cudaStream_t stream);
// claim: the form whose warps claim their CTA's tiles in order (E4M3 codes)
const void* recompress_kernel_ptr(int block, int variant, int fmt, bool claim = false);
const void* gather_kernel_ptr(int block, int fmt);
cudaError_t launch_decompress_shards(const DecompressArgs& a, int block, int fmt, int grid, int P,
                                     cudaStream_t stream);
cudaError_t launch_reduce_recompress(const DecompressArgs& a, int block, int variant, int fmt,
                                     int grid, int batch, cudaStream_t stream);
cudaError_t decompress_fault(unsigned int* bits, bool clear);

// Tensor-core decompress-reduce (block 64 or 128).
size_t decompress_mma_smem_bytes(int block);
const void* decompress_mma_kernel_ptr(int block);
cudaError_t launch_decompress_mma(const DecompressArgs& a, int block, int grid, cudaStream_t stream);
cudaError_t decompress_mma_fault(unsigned int* bits, bool clear);

cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, int64_t n, cudaStream_t st);
cudaError_t launch_e4m3_decode(const uint8_t* in, float* out, int64_t n, cudaStream_t st);
cudaError_t launch_selftest_wait(unsigned long long limit_ns, uint32_t* status, cudaStream_t st);
cudaError_t selftest_fault(unsigned int* bits, bool clear);

}  // namespace taco

// C ABI of the TACO operator: argument checks, shard layout, grid sizing and
// dispatch to the sm_103a kernels. Declarations and contracts are in taco.h.

#include <cmath>
#include <cstdint>
#include <mutex>

#include "taco_launch.h"

namespace taco {

namespace {

constexpr int64_t kMaxElements = int64_t{1} << 40;   // per shard
// Largest target energy E* accepted (2^120): the rotated values of a block
// then stay far inside the fp32 range in every variant (|y| <= sqrt(n E*)),
// and so do the factors the kernels form from alpha. Codes saturate at 448,
// so an E* beyond 448^2 already sends every block to the overflow guard.
constexpr float kMaxTargetEnergy = 0x1p120f;
constexpr int kMaxDevices = 64;

inline size_t pad256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

inline bool valid_block(int block) { return block == 64 || block == 128 || block == 256; }

inline bool valid_variant(int v) {
  return v == TACO_VARIANT_DUAL || v == TACO_VARIANT_ABSMAX || v == TACO_VARIANT_STATIC;
}

inline float static_scale(int block, float target_energy, double q_max = 448.0) {
  return static_cast<float>(std::sqrt(static_cast<double>(block) * target_energy) / q_max);
}

constexpr int kFormats = 2;   // 0 = FP8 E4M3, 1 = INT8 fallback

inline int block_index(int block) { return block == 64 ? 0 : (block == 128 ? 1 : 2); }

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

taco_status check_shape(int64_t N, int64_t h, int block) {
  if (!valid_block(block)) return TACO_ERR_BLOCK;
  if (N < 0 || h <= 0 || h % block != 0) return TACO_ERR_SHAPE;
  if (N > 0 && N > kMaxElements / h) return TACO_ERR_SHAPE;
  return TACO_OK;
}

// Per-device launch facts, filled once per device.
struct DeviceInfo {
  int sms = 0;
  int occ_compress[3][kVariants] = {};
  int occ_decompress[3][kFormats] = {};
  int occ_pw[2][3][kVariants][kFormats] = {};   // producer-warp kernels [mode][block][variant][fmt]
  int occ_recompress[3][kVariants][kFormats] = {};
  int occ_gather[3][kFormats] = {};
  int occ_mma[3][kVariants][kFormats] = {};
  int occ_dmma[2] = {};   // tensor-core decompress, block 64 and 128
};

std::once_flag g_once[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
cudaError_t g_info_err[kMaxDevices];

cudaError_t device_info(const DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_once[dev], [dev]() {
    DeviceInfo& d = g_info[dev];
    cudaError_t err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks[3] = {64, 128, 256};
    const int csmem = static_cast<int>(compress_smem_bytes());
    const int dsmem = static_cast<int>(decompress_smem_bytes());
    for (int m = 0; m < 2 && err == cudaSuccess; ++m)
      for (int b = 0; b < 3 && err == cudaSuccess; ++b)
        for (int v = 0; v < (m == 0 ? 1 : kVariants) && err == cudaSuccess; ++v)
          for (int f = 0; f < kFormats && err == cudaSuccess; ++f) {
            const void* k = decompress_pw_kernel_ptr(m, blocks[b], v, f);
            const int psmem = static_cast<int>(decompress_pw_smem_bytes(blocks[b]));
            err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem);
            if (err == cudaSuccess)
              err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_pw[m][b][v][f], k,
                                                                  kDecompressThreads, psmem);
          }
    for (int b = 0; b < 3 && err == cudaSuccess; ++b) {
      for (int v = 0; v < kVariants && err == cudaSuccess; ++v) {
        const void* k = compress_kernel_ptr(blocks[b], v);
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, csmem);
        if (err == cudaSuccess)
          err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_compress[b][v], k,
                                                              kCompressThreads, csmem);
      }
      for (int f = 0; f < kFormats && err == cudaSuccess; ++f) {
        const void* k = decompress_kernel_ptr(blocks[b], f, false);
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dsmem);
        if (err == cudaSuccess)
          err = cudaFuncSetAttribute(decompress_kernel_ptr(blocks[b], f, true),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, dsmem);
        if (err == cudaSuccess)
          err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_decompress[b][f], k,
                                                              kDecompressThreads, dsmem);
      }
      for (int f = 0; f < kFormats && err == cudaSuccess; ++f) {
        const void* k = gather_kernel_ptr(blocks[b], f);
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dsmem);
        if (err == cudaSuccess)
          err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_gather[b][f], k,
                                                              kDecompressThreads, dsmem);
      }
      for (int v = 0; v < kVariants && err == cudaSuccess; ++v) {
        for (int f = 0; f < kFormats && err == cudaSuccess; ++f) {
          const void* k = compress_mma_kernel_ptr(blocks[b], v, f);
          const int msmem = static_cast<int>(compress_mma_smem_bytes(blocks[b]));
          err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, msmem);
          if (err == cudaSuccess)
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &d.occ_mma[b][v][f], k, compress_mma_threads(blocks[b]), msmem);
        }
      }
      if (err == cudaSuccess && b < 2) {
        const void* k = decompress_mma_kernel_ptr(blocks[b]);
        const int msmem = static_cast<int>(decompress_mma_smem_bytes(blocks[b]));
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, msmem);
        if (err == cudaSuccess)
          err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_dmma[b], k, 320, msmem);
      }
      for (int v = 0; v < kVariants && err == cudaSuccess; ++v) {
        for (int f = 0; f < kFormats && err == cudaSuccess; ++f) {
          const void* k = recompress_kernel_ptr(blocks[b], v, f);
          err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dsmem);
          if (err == cudaSuccess)
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_recompress[b][v][f], k,
                                                                kDecompressThreads, dsmem);
          // the claimed-tile form of the same launch (E4M3 codes)
          if (err == cudaSuccess && f == 0)
            err = cudaFuncSetAttribute(recompress_kernel_ptr(blocks[b], v, f, true),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, dsmem);
        }
      }
    }
    g_info_err[dev] = err;
  });
  if (g_info_err[dev] != cudaSuccess) return g_info_err[dev];
  *out = &g_info[dev];
  return cudaSuccess;
}

struct Layout {
  size_t scales_off, bytes;
};

Layout shard_layout(int64_t N, int64_t h, int block) {
  const size_t elems = static_cast<size_t>(N) * static_cast<size_t>(h);
  const size_t nblk = elems / static_cast<size_t>(block);
  Layout l;
  l.scales_off = pad256(elems);
  l.bytes = l.scales_off + pad256(8 * nblk);
  return l;
}

// CTAs for a CUDA-core kernel of `warps` warps per CTA over `nblocks` blocks:
// enough that every warp gets at least kMinWarpBlocks blocks (its share of a
// grid-stride pass may be a partial tile), so that small tensors still spread
// over many SMs; the caller caps it at the resident CTAs.
constexpr int64_t kMinWarpBlocks = 4;
int64_t ctas_wanted(int64_t nblocks, int warps) {
  const int64_t per_cta = static_cast<int64_t>(warps) * kMinWarpBlocks;
  return (nblocks + per_cta - 1) / per_cta;
}

taco_status decompress_common(const uint8_t* const* shards, int P, int64_t N, int64_t h,
                              int block, void* out, void* stream, int fmt = 0, bool mma = false) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!out) return TACO_ERR_NULL;
  if (!aligned(out, 16)) return TACO_ERR_ALIGN;
  const Layout l = shard_layout(N, h, block);
  const size_t out_bytes = static_cast<size_t>(N) * static_cast<size_t>(h) * 2;
  DecompressArgs a{};
  for (int p = 0; p < P; ++p) {
    if (!shards[p]) return TACO_ERR_NULL;
    if (!aligned(shards[p], 16)) return TACO_ERR_ALIGN;
    if (overlap(shards[p], l.bytes, out, out_bytes)) return TACO_ERR_ARG;
    a.shard[p] = shards[p];
  }
  a.scales_off = l.scales_off;
  a.P = P;
  a.nblocks = N * h / block;
  a.out = static_cast<uint16_t*>(out);
  a.inv_sqrt_n = static_cast<float>(1.0 / std::sqrt(static_cast<double>(block)));

  const DeviceInfo* info = nullptr;
  if (device_info(&info) != cudaSuccess) return TACO_ERR_CUDA;
  if (mma) {
    if (a.nblocks > kMmaMaxBlocks) return TACO_ERR_SHAPE;
    const int occ = info->occ_dmma[block_index(block)];
    if (occ < 1) return TACO_ERR_CUDA;
    int64_t grid = static_cast<int64_t>(info->sms) * occ;
    const int64_t tiles = (a.nblocks + 127) / 128;
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    return launch_decompress_mma(a, block, static_cast<int>(grid), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TACO_OK
               : TACO_ERR_CUDA;
  }
  // the grid of the kernel launch_decompress runs: its own occupancy, and no
  // more CTAs than its smallest share of blocks fills
  const bool pw = decompress_uses_pw(0, block, fmt);
  const int64_t needed = pw ? (a.nblocks + kPwMinBlocksPerCta - 1) / kPwMinBlocksPerCta
                            : ctas_wanted(a.nblocks, kDecompressThreads / 32);
  const int occ = pw ? info->occ_pw[0][block_index(block)][0][fmt] : info->occ_decompress[block_index(block)][fmt];
  if (occ < 1) return TACO_ERR_CUDA;
  int64_t grid = static_cast<int64_t>(info->sms) * occ;
  if (grid > needed) grid = needed;
  if (grid < 1) grid = 1;
  const cudaError_t e = pw ? launch_decompress_pw(a, 0, block, 0, fmt, static_cast<int>(grid), 1,
                                                  static_cast<cudaStream_t>(stream))
                           : launch_decompress(a, block, fmt, static_cast<int>(grid),
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TACO_OK : TACO_ERR_CUDA;
}

taco_status decompress_shards_common(const uint8_t* const* shards, int P, int64_t N, int64_t h,
                                     int block, void* out, void* stream, int fmt = 0) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!out) return TACO_ERR_NULL;
  if (!aligned(out, 16)) return TACO_ERR_ALIGN;
  const Layout l = shard_layout(N, h, block);
  const size_t out_bytes = static_cast<size_t>(P) * N * h * 2;
  DecompressArgs a{};
  for (int p = 0; p < P; ++p) {
    if (!shards[p]) return TACO_ERR_NULL;
    if (!aligned(shards[p], 16)) return TACO_ERR_ALIGN;
    if (overlap(shards[p], l.bytes, out, out_bytes)) return TACO_ERR_ARG;
    a.shard[p] = shards[p];
  }
  a.scales_off = l.scales_off;
  a.P = P;
  a.nblocks = N * h / block;
  a.out = static_cast<uint16_t*>(out);
  a.inv_sqrt_n = static_cast<float>(1.0 / std::sqrt(static_cast<double>(block)));
  const DeviceInfo* info = nullptr;
  if (device_info(&info) != cudaSuccess) return TACO_ERR_CUDA;
  const int64_t needed = ctas_wanted(a.nblocks, kDecompressThreads / 32);
  const int64_t total = static_cast<int64_t>(info->sms) * info->occ_gather[block_index(block)][fmt];
  int64_t gx = (total + P - 1) / P;
  if (gx > needed) gx = needed;
  if (gx < 1) gx = 1;
  if (launch_decompress_shards(a, block, fmt, static_cast<int>(gx), P,
                               static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TACO_ERR_CUDA;
  return TACO_OK;
}

// Y reductions of P shards each in one launch (Y = 1: the single form).
// shards: Y*P pointers, reduction y takes shards[y*P .. y*P+P-1]; the Y
// outputs are consecutive shards from shard_out, headers header_out[0..Y-1].
taco_status reduce_recompress_common(const uint8_t* const* shards, int P, int64_t N, int64_t h,
                                     int block, float target_energy, int variant, void* shard_out,
                                     taco_header* header_out, void* out, void* workspace,
                                     size_t workspace_bytes, void* stream, int fmt = 0, int Y = 1) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || Y < 1 || P * Y > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (Y > 1 && out) return TACO_ERR_ARG;
  if (!valid_variant(variant)) return TACO_ERR_ARG;
  if (!(target_energy > 0.0f) || !(target_energy <= kMaxTargetEnergy)) return TACO_ERR_ARG;
  if (!header_out) return TACO_ERR_NULL;
  if (!workspace || workspace_bytes < Y * kWorkspaceShardStride) return TACO_ERR_WORKSPACE;
  if (!aligned(header_out, 8) || !aligned(workspace, 16)) return TACO_ERR_ALIGN;
  const Layout l = shard_layout(N, h, block);
  const size_t out_bytes = static_cast<size_t>(N) * static_cast<size_t>(h) * 2;
  const size_t rc_bytes = static_cast<size_t>(Y) * l.bytes;
  DecompressArgs a{};
  if (N > 0) {
    if (!shard_out) return TACO_ERR_NULL;
    if (!aligned(shard_out, 16) || (out && !aligned(out, 16))) return TACO_ERR_ALIGN;
    if (out && overlap(out, out_bytes, shard_out, rc_bytes)) return TACO_ERR_ARG;
    for (int p = 0; p < P * Y; ++p) {
      if (!shards[p]) return TACO_ERR_NULL;
      if (!aligned(shards[p], 16)) return TACO_ERR_ALIGN;
      if (overlap(shards[p], l.bytes, shard_out, rc_bytes)) return TACO_ERR_ARG;
      if (out && overlap(shards[p], l.bytes, out, out_bytes)) return TACO_ERR_ARG;
      a.shard[p] = shards[p];
    }
  }
  a.rc_stride = l.bytes;
  a.scales_off = l.scales_off;
  a.P = P;
  a.nblocks = N * h / block;
  a.out = static_cast<uint16_t*>(out);
  a.inv_sqrt_n = static_cast<float>(1.0 / std::sqrt(static_cast<double>(block)));
  a.rc_shard = static_cast<uint8_t*>(shard_out);
  a.rc_header = header_out;
  a.workspace = static_cast<uint8_t*>(workspace);
  a.N = N;
  a.h = h;
  a.target_energy = target_energy;
  a.sqrt_E = static_cast<float>(std::sqrt(static_cast<double>(target_energy)));
  a.sqrt_n = static_cast<float>(std::sqrt(static_cast<double>(block)));
  a.s_static = static_scale(block, target_energy, fmt == 0 ? 448.0 : 127.0);

  const DeviceInfo* info = nullptr;
  if (device_info(&info) != cudaSuccess) return TACO_ERR_CUDA;
  const bool pw = decompress_uses_pw(1, block, fmt);
  const int64_t needed = pw ? (a.nblocks + kPwMinBlocksPerCta - 1) / kPwMinBlocksPerCta
                            : ctas_wanted(a.nblocks, kDecompressThreads / 32);
  const int occ = pw ? info->occ_pw[1][block_index(block)][variant][fmt]
                     : info->occ_recompress[block_index(block)][variant][fmt];
  if (occ < 1) return TACO_ERR_CUDA;
  const int64_t total = static_cast<int64_t>(info->sms) * occ;
  int64_t grid = (total + Y - 1) / Y;
  if (grid > needed) grid = needed;
  if (grid > kMaxCtasPerShard) grid = kMaxCtasPerShard;
  if (grid < 1) grid = 1;
  const cudaError_t e = pw ? launch_decompress_pw(a, 1, block, variant, fmt, static_cast<int>(grid), Y,
                                                  static_cast<cudaStream_t>(stream))
                           : launch_reduce_recompress(a, block, variant, fmt, static_cast<int>(grid), Y,
                                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TACO_OK : TACO_ERR_CUDA;
}

}  // namespace

taco_status check_compress_args(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                                float target_energy, int variant, const void* bundle_out,
                                const taco_header* headers_out, const void* workspace,
                                size_t workspace_bytes) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (!valid_variant(variant)) return TACO_ERR_ARG;
  if (!(target_energy > 0.0f) || !(target_energy <= kMaxTargetEnergy)) return TACO_ERR_ARG;
  if (!headers_out) return TACO_ERR_NULL;
  if (!workspace || workspace_bytes < taco_workspace_bytes(P)) return TACO_ERR_WORKSPACE;
  if (!aligned(headers_out, 8) || !aligned(workspace, 16)) return TACO_ERR_ALIGN;
  if (N > 0) {
    if (!x_bf16 || !bundle_out) return TACO_ERR_NULL;
    if (!aligned(x_bf16, 16) || !aligned(bundle_out, 16)) return TACO_ERR_ALIGN;
    const size_t in_bytes = static_cast<size_t>(P) * N * h * 2;
    if (overlap(x_bf16, in_bytes, bundle_out, P * shard_layout(N, h, block).bytes)) return TACO_ERR_ARG;
  }
  return TACO_OK;
}

namespace {

// Argument checks and kernel arguments shared by both compress entries.
taco_status compress_args(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                          float target_energy, int variant, void* bundle_out,
                          taco_header* headers_out, void* workspace, size_t workspace_bytes,
                          CompressArgs* out) {
  const taco_status st = check_compress_args(x_bf16, P, N, h, block, target_energy, variant,
                                             bundle_out, headers_out, workspace, workspace_bytes);
  if (st != TACO_OK) return st;
  const Layout l = shard_layout(N, h, block);
  const double sqrt_nE = std::sqrt(static_cast<double>(block) * target_energy);

  CompressArgs& a = *out;
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.shard_elems = N * h;
  a.nblocks = N * h / block;
  a.bundle = static_cast<uint8_t*>(bundle_out);
  a.shard_bytes = l.bytes;
  a.scales_off = l.scales_off;
  a.headers = headers_out;
  a.workspace = static_cast<uint8_t*>(workspace);
  a.N = N;
  a.h = h;
  a.target_energy = target_energy;
  a.sqrt_nE = static_cast<float>(sqrt_nE);
  a.inv_sqrt_n = static_cast<float>(1.0 / std::sqrt(static_cast<double>(block)));
  a.s_static = static_scale(block, target_energy);
  a.q_max = 448.0f;
  return TACO_OK;
}

// The tensor-core compress for both code formats (0 = E4M3, 1 = INT8).
taco_status compress_mma_common(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                                float target_energy, int variant, void* bundle_out,
                                taco_header* headers_out, void* workspace, size_t workspace_bytes,
                                void* stream, int fmt) {
  CompressArgs a{};
  taco_status st = compress_args(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                                 headers_out, workspace, workspace_bytes, &a);
  if (st != TACO_OK) return st;
  if (a.nblocks > kMmaMaxBlocks) return TACO_ERR_SHAPE;
  const double n_sqrtE = block * std::sqrt(static_cast<double>(target_energy));   // finite
  a.n_sqrtE = static_cast<float>(n_sqrtE);
  if (fmt == 1) {
    a.s_static = static_scale(block, target_energy, 127.0);
    a.q_max = 127.0f;
  }

  const DeviceInfo* info = nullptr;
  if (device_info(&info) != cudaSuccess) return TACO_ERR_CUDA;
  if (N == 0) {
    // nothing to rotate or encode: one CTA per shard of the CUDA-core kernel
    // writes the headers (its code loop is empty)
    return launch_compress(a, block, variant, 1, P, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? TACO_OK
               : TACO_ERR_CUDA;
  }
  const int occ = info->occ_mma[block_index(block)][variant][fmt];
  if (occ < 1) return TACO_ERR_CUDA;
  const int64_t tiles = (a.nblocks + 127) / 128;
  int64_t gx = static_cast<int64_t>(info->sms) * occ / P;
  if (gx > tiles) gx = tiles;
  if (gx > kMaxCtasPerShard) gx = kMaxCtasPerShard;
  if (gx < 1) gx = 1;
  if (launch_compress_mma(a, block, variant, fmt, static_cast<int>(gx), P,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TACO_ERR_CUDA;
  return TACO_OK;
}

}  // namespace
}  // namespace taco

using namespace taco;

extern "C" {

size_t taco_shard_bytes(int64_t N, int64_t h, int block) {
  if (check_shape(N, h, block) != TACO_OK) return 0;
  return shard_layout(N, h, block).bytes;
}

size_t taco_shard_scales_offset(int64_t N, int64_t h, int block) {
  if (check_shape(N, h, block) != TACO_OK) return 0;
  return shard_layout(N, h, block).scales_off;
}

size_t taco_workspace_bytes(int P) {
  if (P < 1 || P > TACO_MAX_SHARDS) return 0;
  return static_cast<size_t>(P) * kWorkspaceShardStride;
}

taco_status taco_compress_shards_mma(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                                     float target_energy, int variant, void* bundle_out,
                                     taco_header* headers_out, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return compress_mma_common(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                             headers_out, workspace, workspace_bytes, stream, 0);
}

taco_status taco_compress_shards_int8(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                                      float target_energy, int variant, void* bundle_out,
                                      taco_header* headers_out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return compress_mma_common(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                             headers_out, workspace, workspace_bytes, stream, 1);
}

taco_status taco_compress_shards(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                                 float target_energy, int variant, void* bundle_out,
                                 taco_header* headers_out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  // the tensor-core kernel wherever its tensor copies can address the shard
  // (faster on every measured shape), the CUDA-core FWHT beyond that
  CompressArgs a{};
  const taco_status st = compress_args(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                                       headers_out, workspace, workspace_bytes, &a);
  if (st != TACO_OK) return st;
  if (a.nblocks > kMmaMaxBlocks)
    return taco_compress_shards_fwht(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                                     headers_out, workspace, workspace_bytes, stream);
  return compress_mma_common(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                             headers_out, workspace, workspace_bytes, stream, 0);
}

taco_status taco_compress_shards_fwht(const void* x_bf16, int P, int64_t N, int64_t h, int block,
                                      float target_energy, int variant, void* bundle_out,
                                      taco_header* headers_out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  CompressArgs a{};
  taco_status st = compress_args(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                                 headers_out, workspace, workspace_bytes, &a);
  if (st != TACO_OK) return st;
  const DeviceInfo* info = nullptr;
  if (device_info(&info) != cudaSuccess) return TACO_ERR_CUDA;
  const int64_t needed = ctas_wanted(a.nblocks, kCompressThreads / 32);
  const int64_t total = static_cast<int64_t>(info->sms) * info->occ_compress[block_index(block)][variant];
  int64_t gx = (total + P - 1) / P;
  if (gx > needed) gx = needed;
  if (gx > kMaxCtasPerShard) gx = kMaxCtasPerShard;
  if (gx < 1) gx = 1;
  if (launch_compress(a, block, variant, static_cast<int>(gx), P, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return TACO_ERR_CUDA;
  return TACO_OK;
}


taco_status taco_compress(const void* x_bf16, int64_t N, int64_t h, int block, float target_energy,
                          int variant, void* shard_out, taco_header* header_out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return taco_compress_shards(x_bf16, 1, N, h, block, target_energy, variant, shard_out,
                              header_out, workspace, workspace_bytes, stream);
}

taco_status taco_decompress_reduce(const void* bundle, int P, int64_t N, int64_t h, int block,
                                   void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!bundle) return TACO_ERR_NULL;
  const size_t sb = shard_layout(N, h, block).bytes;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(bundle) + p * sb;
  return decompress_common(ptrs, P, N, h, block, out_bf16, stream);
}

taco_status taco_decompress_reduce_int8(const void* bundle, int P, int64_t N, int64_t h, int block,
                                        void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!bundle) return TACO_ERR_NULL;
  const size_t sb = shard_layout(N, h, block).bytes;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(bundle) + p * sb;
  return decompress_common(ptrs, P, N, h, block, out_bf16, stream, 1);
}

taco_status taco_decompress_reduce_mma(const void* bundle, int P, int64_t N, int64_t h, int block,
                                       void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (block == 256) return TACO_ERR_BLOCK;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!bundle) return TACO_ERR_NULL;
  const size_t sb = shard_layout(N, h, block).bytes;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(bundle) + p * sb;
  return decompress_common(ptrs, P, N, h, block, out_bf16, stream, 0, true);
}

taco_status taco_decompress_reduce_mma_ptrs(const void* const* shards, int P, int64_t N, int64_t h,
                                            int block, void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (block == 256) return TACO_ERR_BLOCK;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!shards) return TACO_ERR_NULL;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(shards[p]);
  return decompress_common(ptrs, P, N, h, block, out_bf16, stream, 0, true);
}

taco_status taco_decompress_reduce_ptrs(const void* const* shards, int P, int64_t N, int64_t h,
                                        int block, void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!shards) return TACO_ERR_NULL;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(shards[p]);
  return decompress_common(ptrs, P, N, h, block, out_bf16, stream);
}

taco_status taco_decompress_shards(const void* bundle, int P, int64_t N, int64_t h, int block,
                                   void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!bundle) return TACO_ERR_NULL;
  const size_t sb = shard_layout(N, h, block).bytes;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(bundle) + p * sb;
  return decompress_shards_common(ptrs, P, N, h, block, out_bf16, stream);
}

taco_status taco_decompress_shards_ptrs(const void* const* shards, int P, int64_t N, int64_t h,
                                        int block, void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!shards) return TACO_ERR_NULL;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(shards[p]);
  return decompress_shards_common(ptrs, P, N, h, block, out_bf16, stream);
}

taco_status taco_reduce_recompress(const void* bundle, int P, int64_t N, int64_t h, int block,
                                   float target_energy, int variant, void* shard_out,
                                   taco_header* header_out, void* out_bf16, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N > 0 && !bundle) return TACO_ERR_NULL;
  const size_t sb = shard_layout(N, h, block).bytes;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(bundle) + p * sb;
  return reduce_recompress_common(ptrs, P, N, h, block, target_energy, variant, shard_out,
                                  header_out, out_bf16, workspace, workspace_bytes, stream);
}

taco_status taco_reduce_recompress_ptrs(const void* const* shards, int P, int64_t N, int64_t h,
                                        int block, float target_energy, int variant,
                                        void* shard_out, taco_header* header_out, void* out_bf16,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (!shards) return TACO_ERR_NULL;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(shards[p]);
  return reduce_recompress_common(ptrs, P, N, h, block, target_energy, variant, shard_out,
                                  header_out, out_bf16, workspace, workspace_bytes, stream);
}

taco_status taco_reduce_recompress_int8_ptrs(const void* const* shards, int P, int64_t N,
                                             int64_t h, int block, float target_energy,
                                             int variant, void* shard_out,
                                             taco_header* header_out, void* out_bf16,
                                             void* workspace, size_t workspace_bytes,
                                             void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (!shards) return TACO_ERR_NULL;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(shards[p]);
  return reduce_recompress_common(ptrs, P, N, h, block, target_energy, variant, shard_out,
                                  header_out, out_bf16, workspace, workspace_bytes, stream, 1);
}

taco_status taco_reduce_recompress_batched_ptrs(const void* const* shards, int Y, int P, int64_t N,
                                                int64_t h, int block, float target_energy,
                                                int variant, int code_format, void* shards_out,
                                                taco_header* headers_out, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (Y < 1 || P < 1 || static_cast<int64_t>(Y) * P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (code_format != TACO_FORMAT_E4M3 && code_format != TACO_FORMAT_INT8) return TACO_ERR_ARG;
  if (!shards) return TACO_ERR_NULL;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < Y * P; ++p) ptrs[p] = static_cast<const uint8_t*>(shards[p]);
  return reduce_recompress_common(ptrs, P, N, h, block, target_energy, variant, shards_out,
                                  headers_out, nullptr, workspace, workspace_bytes, stream,
                                  code_format, Y);
}

taco_status taco_decompress_shards_int8_ptrs(const void* const* shards, int P, int64_t N,
                                             int64_t h, int block, void* out_bf16, void* stream) {
  taco_status st = check_shape(N, h, block);
  if (st != TACO_OK) return st;
  if (P < 1 || P > TACO_MAX_SHARDS) return TACO_ERR_ARG;
  if (N == 0) return TACO_OK;
  if (!shards) return TACO_ERR_NULL;
  const uint8_t* ptrs[TACO_MAX_SHARDS];
  for (int p = 0; p < P; ++p) ptrs[p] = static_cast<const uint8_t*>(shards[p]);
  return decompress_shards_common(ptrs, P, N, h, block, out_bf16, stream, 1);
}

taco_status taco_e4m3_encode_f32(const float* in, uint8_t* out, int64_t n, void* stream) {
  if (n < 0) return TACO_ERR_SHAPE;
  if (n == 0) return TACO_OK;
  if (!in || !out) return TACO_ERR_NULL;
  if (!aligned(in, 4)) return TACO_ERR_ALIGN;
  return launch_e4m3_encode(in, out, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TACO_OK
             : TACO_ERR_CUDA;
}

taco_status taco_e4m3_decode_f32(const uint8_t* in, float* out, int64_t n, void* stream) {
  if (n < 0) return TACO_ERR_SHAPE;
  if (n == 0) return TACO_OK;
  if (!in || !out) return TACO_ERR_NULL;
  if (!aligned(out, 4)) return TACO_ERR_ALIGN;
  return launch_e4m3_decode(in, out, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TACO_OK
             : TACO_ERR_CUDA;
}

taco_status taco_get_fault(uint32_t* bits, int clear) {
  if (!bits) return TACO_ERR_NULL;
  unsigned int c = 0, d = 0, t = 0, m = 0, dm = 0, dp = 0;
  if (compress_fault(&c, clear != 0) != cudaSuccess) return TACO_ERR_CUDA;
  if (decompress_pw_fault(&dp, clear != 0) != cudaSuccess) return TACO_ERR_CUDA;
  if (compress_mma_fault(&m, clear != 0) != cudaSuccess) return TACO_ERR_CUDA;
  if (decompress_mma_fault(&dm, clear != 0) != cudaSuccess) return TACO_ERR_CUDA;
  if (decompress_fault(&d, clear != 0) != cudaSuccess) return TACO_ERR_CUDA;
  if (selftest_fault(&t, clear != 0) != cudaSuccess) return TACO_ERR_CUDA;
  *bits = c | d | t | m | dm | dp;
  return TACO_OK;
}

taco_status taco_selftest_wait_timeout(uint64_t limit_ns, uint32_t* status_dev, void* stream) {
  if (!status_dev) return TACO_ERR_NULL;
  if (!aligned(status_dev, 4)) return TACO_ERR_ALIGN;
  if (limit_ns == 0 || limit_ns > 2000000000ull) return TACO_ERR_ARG;
  return launch_selftest_wait(limit_ns, status_dev, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TACO_OK
             : TACO_ERR_CUDA;
}

const char* taco_status_string(taco_status s) {
  switch (s) {
    case TACO_OK: return "ok";
    case TACO_ERR_NULL: return "null pointer";
    case TACO_ERR_SHAPE: return "bad shape (N < 0, h <= 0, h % block != 0 or too large)";
    case TACO_ERR_BLOCK: return "block size must be 64, 128 or 256";
    case TACO_ERR_ALIGN: return "pointer not aligned (tensors and bundles need 16 bytes)";
    case TACO_ERR_ARG: return "bad argument (target energy, P, variant or overlapping buffers)";
    case TACO_ERR_CUDA: return "CUDA error";
    case TACO_ERR_WORKSPACE: return "workspace missing or smaller than taco_workspace_bytes";
  }
  return "unknown status";
}

int taco_abi_version(void) { return TACO_ABI_VERSION; }

}  // extern "C"

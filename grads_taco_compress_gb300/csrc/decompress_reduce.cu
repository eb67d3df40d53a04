// TACO fused decompress-reduce kernel for sm_103a.
//
// Reconstruction with the two scales ("TACO: Efficient Communication
// Compression of Intermediate Tensors ...", gist.science pt summary, §2.B.2)
// fused with the reduce of the ReduceScatter half of the two-shot AllReduce
// (same page, §2.B.3), for P shards that share the block partition:
//   z      = sum_p (s_p / alpha_p / sqrt(n)) dec(q_p)     (fp32, rotated domain)
//   x_hat  = bf16( H_n z )                                 (one inverse rotation)
// H_n / sqrt(n) is symmetric and orthogonal, so it is its own inverse, and the
// sum can be taken before the rotation because the rotation is linear.
// Each thread owns the same 8*CH elements of a block as in compress; per shard
// it issues CH 8-byte code loads and two scalar scale loads (shared by the
// block's lanes), decodes E4M3 pairs with cvt.rn.f16x2.e4m3x2 and
// accumulates with one FMA per element. The grid is persistent over warp
// tiles.

#include "taco_device.cuh"
#include "taco_launch.h"

namespace taco {

namespace {

template <int NB, int CH>
__global__ void __launch_bounds__(kDecompressThreads)
decompress_reduce_kernel(DecompressArgs a) {
  constexpr int LPB = NB / (8 * CH);
  constexpr int BPT = 32 / LPB;
  static_assert(LPB >= 1 && LPB <= 32 && (LPB & (LPB - 1)) == 0, "bad split");

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = lane & (LPB - 1);
  const int sub = lane / LPB;

  const int64_t nblocks = a.nblocks;
  const int64_t tiles = (nblocks + BPT - 1) / BPT;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kDecompressThreads / 32);

  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * (kDecompressThreads / 32) + warp;
       tile < tiles; tile += stride) {
    const int64_t b = tile * BPT + sub;
    const bool valid = b < nblocks;
    const int64_t bb = valid ? b : 0;

    float z[CH][8];
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i) z[c][i] = 0.f;

#pragma unroll 2
    for (int p = 0; p < a.P; ++p) {
      const uint8_t* base = a.shard[p];
      uint2 q[CH];
#pragma unroll
      for (int c = 0; c < CH; ++c)
        q[c] = valid ? ld_stream_v2(base + bb * NB + 8 * (j + LPB * c)) : make_uint2(0, 0);
      const float al = ld_stream_f32(reinterpret_cast<const float*>(base + a.alpha_off) + bb);
      const float sc = ld_stream_f32(reinterpret_cast<const float*>(base + a.s_off) + bb);
      const float d = sc * __frcp_rn(al) * a.inv_sqrt_n;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const float2 f0 = e4m3x2_to_f32(q[c].x & 0xffffu);
        const float2 f1 = e4m3x2_to_f32(q[c].x >> 16);
        const float2 f2 = e4m3x2_to_f32(q[c].y & 0xffffu);
        const float2 f3 = e4m3x2_to_f32(q[c].y >> 16);
        z[c][0] = fmaf(d, f0.x, z[c][0]); z[c][1] = fmaf(d, f0.y, z[c][1]);
        z[c][2] = fmaf(d, f1.x, z[c][2]); z[c][3] = fmaf(d, f1.y, z[c][3]);
        z[c][4] = fmaf(d, f2.x, z[c][4]); z[c][5] = fmaf(d, f2.y, z[c][5]);
        z[c][6] = fmaf(d, f3.x, z[c][6]); z[c][7] = fmaf(d, f3.y, z[c][7]);
      }
    }

    fwht_in_registers<CH>(z);
    fwht_across_lanes<CH, LPB>(z, j);

    if (valid) {
      uint16_t* op = a.out + b * NB;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        uint4 w;
        w.x = pack_bf16x2(z[c][0], z[c][1]);
        w.y = pack_bf16x2(z[c][2], z[c][3]);
        w.z = pack_bf16x2(z[c][4], z[c][5]);
        w.w = pack_bf16x2(z[c][6], z[c][7]);
        *reinterpret_cast<uint4*>(op + 8 * (j + LPB * c)) = w;
      }
    }
  }
}

}  // namespace

constexpr int kDecompressCH = 4;

int decompress_tile_blocks(int block) { return 32 / (block / (8 * kDecompressCH)); }

const void* decompress_kernel_ptr(int block) {
  switch (block) {
    case 64: return reinterpret_cast<const void*>(decompress_reduce_kernel<64, kDecompressCH>);
    case 128: return reinterpret_cast<const void*>(decompress_reduce_kernel<128, kDecompressCH>);
    default: return reinterpret_cast<const void*>(decompress_reduce_kernel<256, kDecompressCH>);
  }
}

cudaError_t launch_decompress(const DecompressArgs& a, int block, int grid, cudaStream_t stream) {
  switch (block) {
    case 64:
      decompress_reduce_kernel<64, kDecompressCH><<<grid, kDecompressThreads, 0, stream>>>(a);
      break;
    case 128:
      decompress_reduce_kernel<128, kDecompressCH><<<grid, kDecompressThreads, 0, stream>>>(a);
      break;
    default:
      decompress_reduce_kernel<256, kDecompressCH><<<grid, kDecompressThreads, 0, stream>>>(a);
      break;
  }
  return cudaGetLastError();
}

}  // namespace taco

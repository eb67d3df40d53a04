// TACO fused compress kernel for sm_103a.
//
// One launch does every step of the operator ("TACO: Efficient Communication
// Compression of Intermediate Tensors ...", gist.science pt summary, §2.B.3:
// energy, ASH and DS quantisation fused in one kernel, no intermediate
// global-memory round trip):
//   load bf16 (16-byte streaming loads) -> block energy (fp32, lane shuffles)
//   -> FWHT of the raw block in registers/shuffles (the rotation is linear,
//   so alpha is applied afterwards together with 1/sqrt(n) and 1/s)
//   -> alpha = sqrt(E*/E), s = max(1, alpha/sqrt(n) * max|Hx| / 448)
//   -> E4M3 codes with cvt.rn.satfinite (8-byte stores), alpha and s stores
//   -> per-tensor header through per-CTA partials and a last-CTA reduction.
// The grid is persistent: gridDim.y = shard, gridDim.x CTAs per shard, each
// warp walking warp tiles (32/LPB blocks) with a stride of the whole grid row,
// prefetching the next tile's loads before working on the current one.

#include <cmath>

#include "taco_device.cuh"
#include "taco_launch.h"

namespace taco {

namespace {

template <int NB, int CH>
struct CompressShape {
  static constexpr int kLPB = NB / (8 * CH);       // lanes per block
  static constexpr int kBPT = 32 / kLPB;           // blocks per warp tile
  static_assert(kLPB >= 1 && kLPB <= 32 && (kLPB & (kLPB - 1)) == 0, "bad split");
};

template <int CH, int LPB>
__device__ __forceinline__ void load_tile(const uint16_t* __restrict__ x, int64_t b, bool valid,
                                          int j, uint4 (&raw)[CH]) {
  const uint16_t* blk = x + (valid ? b : 0) * (8 * CH * LPB);
#pragma unroll
  for (int v = 0; v < CH; ++v) {
    raw[v] = valid ? ld_stream_v4(blk + 8 * (j + LPB * v)) : make_uint4(0, 0, 0, 0);
  }
}

template <int NB, int CH, int VARIANT>
__global__ void __launch_bounds__(kCompressThreads)
compress_kernel(CompressArgs a) {
  using S = CompressShape<NB, CH>;
  constexpr int LPB = S::kLPB;
  constexpr int BPT = S::kBPT;

  const int shard = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = lane & (LPB - 1);                   // lane inside its block
  const int sub = lane / LPB;                       // block inside the tile

  const uint16_t* __restrict__ x = a.x + static_cast<int64_t>(shard) * a.shard_elems;
  uint8_t* shard_base = a.bundle + static_cast<size_t>(shard) * a.shard_bytes;
  uint8_t* __restrict__ codes = shard_base;
  float* __restrict__ alpha_out = reinterpret_cast<float*>(shard_base + a.alpha_off);
  float* __restrict__ s_out = reinterpret_cast<float*>(shard_base + a.s_off);

  const int64_t nblocks = a.nblocks;
  const int64_t tiles = (nblocks + BPT - 1) / BPT;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kCompressThreads / 32);
  int64_t tile = static_cast<int64_t>(blockIdx.x) * (kCompressThreads / 32) + warp;

  float part_smax = 0.0f;   // header partials of this thread (lane j == 0 only)
  uint32_t part_cnt = 0;

  uint4 raw[CH];
  {
    const int64_t b = tile * BPT + sub;
    load_tile<CH, LPB>(x, b, tile < tiles && b < nblocks, j, raw);
  }

  for (; tile < tiles; tile += stride) {
    const int64_t b = tile * BPT + sub;
    const bool valid = b < nblocks;

    // Prefetch the next tile of this warp.
    uint4 nxt[CH];
    {
      const int64_t tn = tile + stride;
      const int64_t bn = tn * BPT + sub;
      load_tile<CH, LPB>(x, bn, tn < tiles && bn < nblocks, j, nxt);
    }

    float v[CH][8];
#pragma unroll
    for (int c = 0; c < CH; ++c) unpack_bf16x8(raw[c], v[c]);

    // Block energy (sum of squares; E = e / NB). Four partial sums, then the
    // lanes of the block.
    float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      e0 = fmaf(v[c][0], v[c][0], e0); e1 = fmaf(v[c][1], v[c][1], e1);
      e2 = fmaf(v[c][2], v[c][2], e2); e3 = fmaf(v[c][3], v[c][3], e3);
      e0 = fmaf(v[c][4], v[c][4], e0); e1 = fmaf(v[c][5], v[c][5], e1);
      e2 = fmaf(v[c][6], v[c][6], e2); e3 = fmaf(v[c][7], v[c][7], e3);
    }
    const float e = block_sum<LPB>((e0 + e1) + (e2 + e3));

    // Rotation of the raw block: t = H x.
    fwht_in_registers<CH>(v);
    fwht_across_lanes<CH, LPB>(v, j);

    float tmax = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i) tmax = fmaxf(tmax, fabsf(v[c][i]));
    tmax = block_max<LPB>(tmax);

    // alpha = sqrt(E*/E) = sqrt(n E*) / sqrt(e): reciprocal square root with
    // one Newton step (error about one ulp), 1 for an all-zero block.
    float alpha = 1.0f;
    if (e > 0.f) {
      float r = rsqrtf(e);
      const float hr = 0.5f * e * r;
      r = fmaf(fmaf(-hr, r, 0.5f), r, r);
      alpha = a.sqrt_nE * r;
    }
    const float cscale = alpha * a.inv_sqrt_n;        // y = cscale * t
    const float amax = cscale * tmax;
    float s;
    if (VARIANT == 0) {
      s = fmaxf(1.0f, amax * (1.0f / 448.0f));
    } else {
      s = amax > 0.f ? amax * (1.0f / 448.0f) : 1.0f;
    }
    const float g = (s == 1.0f) ? cscale : cscale / s;  // code value = g * t

    if (valid) {
      uint8_t* cp = codes + b * NB;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        uint2 w;
        w.x = e4m3x4_from_f32(v[c][0] * g, v[c][1] * g, v[c][2] * g, v[c][3] * g);
        w.y = e4m3x4_from_f32(v[c][4] * g, v[c][5] * g, v[c][6] * g, v[c][7] * g);
        *reinterpret_cast<uint2*>(cp + 8 * (j + LPB * c)) = w;
      }
      if (j == 0) {
        alpha_out[b] = alpha;
        s_out[b] = s;
        part_smax = fmaxf(part_smax, s);
        part_cnt += (s > 1.0f) ? 1u : 0u;
      }
    }

#pragma unroll
    for (int c = 0; c < CH; ++c) raw[c] = nxt[c];
  }

  // ---- per-tensor header: CTA reduction, then the last CTA of the shard ----
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    part_smax = fmaxf(part_smax, __shfl_xor_sync(kFullMask, part_smax, m));
    part_cnt += __shfl_xor_sync(kFullMask, part_cnt, m);
  }
  __shared__ float sh_max[kCompressThreads / 32];
  __shared__ uint32_t sh_cnt[kCompressThreads / 32];
  __shared__ bool sh_last;
  if (lane == 0) {
    sh_max[warp] = part_smax;
    sh_cnt[warp] = part_cnt;
  }
  __syncthreads();

  uint32_t* counter = reinterpret_cast<uint32_t*>(a.workspace + shard * kWorkspaceShardStride);
  float2* partials = reinterpret_cast<float2*>(a.workspace + shard * kWorkspaceShardStride + 16);
  if (threadIdx.x == 0) {
    float m = 0.f;
    uint32_t n = 0;
    for (int w = 0; w < kCompressThreads / 32; ++w) {
      m = fmaxf(m, sh_max[w]);
      n += sh_cnt[w];
    }
    partials[blockIdx.x] = make_float2(m, __uint_as_float(n));
    __threadfence();
    const uint32_t arrived = atomicAdd(counter, 1u);
    sh_last = (arrived == gridDim.x - 1);
  }
  __syncthreads();

  if (sh_last) {
    __threadfence();
    float m = 0.f;
    uint32_t n = 0;
    for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kCompressThreads) {
      const float2 p = __ldcg(partials + i);
      m = fmaxf(m, p.x);
      n += __float_as_uint(p.y);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
      n += __shfl_xor_sync(kFullMask, n, o);
    }
    __syncthreads();
    if (lane == 0) {
      sh_max[warp] = m;
      sh_cnt[warp] = n;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kCompressThreads / 32; ++w) {
        m = fmaxf(m, sh_max[w]);
        n += sh_cnt[w];
      }
      taco_header* hd = a.headers + shard;
      hd->N = a.N;
      hd->h = a.h;
      hd->block = NB;
      hd->variant = VARIANT;
      hd->target_energy = a.target_energy;
      hd->q_max = 448.0f;
      hd->s_max = m;
      hd->n_clamped = n;
      *counter = 0u;   // leave the workspace zero-filled for the next call
    }
  }
}

template <int NB, int CH>
cudaError_t launch_nb(const CompressArgs& a, int variant, int grid_x, int P, cudaStream_t st) {
  const dim3 grid(grid_x, P);
  if (variant == 0) {
    compress_kernel<NB, CH, 0><<<grid, kCompressThreads, 0, st>>>(a);
  } else {
    compress_kernel<NB, CH, 1><<<grid, kCompressThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

template <int NB, int CH>
const void* kernel_ptr(int variant) {
  return variant == 0 ? reinterpret_cast<const void*>(compress_kernel<NB, CH, 0>)
                      : reinterpret_cast<const void*>(compress_kernel<NB, CH, 1>);
}

}  // namespace

// Chunks of 8 elements held per thread, per block size.
constexpr int kCompressCH = 4;

int compress_tile_blocks(int block) { return 32 / (block / (8 * kCompressCH)); }

const void* compress_kernel_ptr(int block, int variant) {
  switch (block) {
    case 64: return kernel_ptr<64, kCompressCH>(variant);
    case 128: return kernel_ptr<128, kCompressCH>(variant);
    default: return kernel_ptr<256, kCompressCH>(variant);
  }
}

cudaError_t launch_compress(const CompressArgs& a, int block, int variant, int grid_x, int P,
                            cudaStream_t stream) {
  switch (block) {
    case 64: return launch_nb<64, kCompressCH>(a, variant, grid_x, P, stream);
    case 128: return launch_nb<128, kCompressCH>(a, variant, grid_x, P, stream);
    default: return launch_nb<256, kCompressCH>(a, variant, grid_x, P, stream);
  }
}

}  // namespace taco

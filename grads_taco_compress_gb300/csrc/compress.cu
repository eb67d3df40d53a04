// TACO fused compress kernel for sm_103a with the rotation as a CUDA-core
// FWHT (taco_compress_shards, taco_compress, taco_compress_shards_noalloc;
// compress_mma.cu holds the tensor-core kernel).
//
// One launch does every step of the operator ("TACO: Efficient Communication
// Compression of Intermediate Tensors ...", gist.science pt summary, §2.B.3:
// energy, ASH and DS quantisation fused in one kernel, no intermediate
// global-memory round trip):
//   TMA bulk copy of the bf16 tile into shared memory -> block energy (fp32,
//   packed FMAs, lane shuffles; a block far from 1 is redone scaled by a
//   power of two, far_tile) -> FWHT of the raw block in registers and
//   shuffles (the rotation is linear, so alpha is applied afterwards together
//   with 1/sqrt(n) and 1/s) -> alpha = sqrt(E*/E), s = max(1, alpha/sqrt(n) *
//   max|Hx| / 448) (ABSMAX: without the floor; STATIC: the per-tensor
//   sqrt(n E*)/448) -> E4M3 codes with cvt.rn.satfinite, written into the
//   tile's shared-memory stage and stored with one TMA bulk store per tile,
//   one (alpha, s) pair store per block -> per-tensor header through running
//   totals in the workspace, finished by the last CTA to arrive.
// Grid: gridDim.y = shard, gridDim.x persistent CTAs per shard. Each warp
// walks warp tiles (2048 elements, 32/LPB blocks) in grid-stride rounds and
// then an even share of the blocks left over (WarpWork), keeping
// kCompressStages tiles in flight: lane 0 issues a 1-D
// cp.async.bulk per tile into the warp's ring of shared-memory stages, each
// completed on its own mbarrier; all lanes wait (bounded in time) and read
// their chunks; the stage then holds the tile's codes until their bulk store
// has read them, and is refilled one tile later.

#include <cmath>

#include "taco_device.cuh"
#include "taco_launch.h"

namespace taco {

namespace {

__device__ unsigned int g_compress_fault;

// The warp's tile again, for a warp with at least one non-zero block whose
// sum of squares is not a trusted fp32 number (subnormal squares, or a sum or
// transform that may overflow). Runs after the common path has written its
// codes into the stage (which no longer holds x), so every block of the tile
// is read again from global memory (`xb`: the tile's first block) and scaled
// by 2^-k (k the lane's: the exponent of the block's max |t| from the common
// path, 128 if that overflowed; 0 for the blocks that were in range, which
// repeats their computation exactly); its energy, alpha (2^-k put back, kept
// in [2^-126, 2^126]), s and codes are computed as in the kernel and the
// codes overwrite the stage's. Returns (alpha, s) of the lane's block. Rare,
// so it is a call of its own: the common path keeps its registers.
template <int NB, int VARIANT>
__device__ __noinline__ float2 far_tile(const uint16_t* __restrict__ xb, bool valid, uint32_t stage, int sub,
                                        int j, int cx, int k, float sqrt_nE, float inv_sqrt_n, float s_static) {
  constexpr int LPB = NB / 64;
  const int nk = -k, nk1 = nk >> 1;                   // 2^-k = 2^nk1 2^(nk - nk1), both normal
  const f2 s1{exp2i(nk1), exp2i(nk1)}, s2{exp2i(nk - nk1), exp2i(nk - nk1)};
  f2 v[kCH][4];
  const uint4* src = reinterpret_cast<const uint4*>(xb + sub * NB);
#pragma unroll
  for (int q = 0; q < kCH; ++q) {
    const uint4 r = valid ? __ldg(src + j + LPB * (q ^ cx)) : make_uint4(0u, 0u, 0u, 0u);
    v[q][0] = mul2(mul2(f2{bf16_lo(r.x), bf16_hi(r.x)}, s1), s2);
    v[q][1] = mul2(mul2(f2{bf16_lo(r.y), bf16_hi(r.y)}, s1), s2);
    v[q][2] = mul2(mul2(f2{bf16_lo(r.z), bf16_hi(r.z)}, s1), s2);
    v[q][3] = mul2(mul2(f2{bf16_lo(r.w), bf16_hi(r.w)}, s1), s2);
  }
  f2 ea[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int q = 0; q < kCH; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) ea[i] = fma2(v[q][i], v[q][i], ea[i]);
  const f2 e01 = add2(ea[0], ea[1]), e23 = add2(ea[2], ea[3]);
  const float e = block_sum<LPB>((e01.x + e01.y) + (e23.x + e23.y));
  float r = rsqrtf(e);
  r = fmaf(fmaf(-0.5f * e * r, r, 0.5f), r, r);
  const float alpha = (e > 0.f) ? clamp_alpha(sqrt_nE * r * s1.x * s2.x) : 1.0f;
  // y = alpha 2^k t' / sqrt(n): 2^k undoes the scaling of the block
  const float cscale = alpha * exp2i(-nk1) * exp2i(nk1 - nk) * inv_sqrt_n;
  fwht_in_registers<kCH>(v, cx);
  fwht_across_lanes<kCH, LPB>(v, j);
  float hi = -INFINITY, lo = INFINITY;
#pragma unroll
  for (int q = 0; q < kCH; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      hi = max3(hi, v[q][i].x, v[q][i].y);
      lo = min3(lo, v[q][i].x, v[q][i].y);
    }
  const float amax = cscale * block_max<LPB>(fmaxf(hi, -lo));
  const float sc = (VARIANT == 0)   ? fmaxf(1.0f, amax * (1.0f / 448.0f))
                   : (VARIANT == 1) ? (amax > 0.f ? amax * (1.0f / 448.0f) : 1.0f)
                                    : s_static;
  const f2 g2{__fdividef(cscale, sc), __fdividef(cscale, sc)};
  const uint32_t cbase = stage + sub * NB;
#pragma unroll
  for (int q = 0; q < kCH; ++q) {
    const f2 y0 = mul2(v[q][0], g2), y1 = mul2(v[q][1], g2);
    const f2 y2 = mul2(v[q][2], g2), y3 = mul2(v[q][3], g2);
    uint2 w;
    w.x = e4m3x4_from_f32(y0.x, y0.y, y1.x, y1.y);
    w.y = e4m3x4_from_f32(y2.x, y2.y, y3.x, y3.y);
    sts64(cbase + 8 * (j + LPB * (q ^ cx)), w);
  }
  return make_float2(alpha, sc);
}

template <int NB, int VARIANT>
__global__ void __launch_bounds__(kCompressThreads, kCompressMinBlocks)
compress_kernel(CompressArgs a) {
  constexpr int LPB = NB / 64;                 // lanes per block
  constexpr int BPT = 32 / LPB;                // blocks per warp tile
  constexpr int D = kCompressStages;
  constexpr int WARPS = kCompressThreads / 32;
  constexpr uint32_t TILE_BYTES = kTileElems * 2;
  static_assert(LPB >= 1 && LPB <= 4, "block size");

  extern __shared__ __align__(128) unsigned char smem[];

  const int shard = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = lane & (LPB - 1);              // lane inside its block
  const int sub = lane / LPB;                  // block inside the tile
  const int cx = sub & (kCH - 1);              // chunk-slot swizzle

  const uint32_t stage0 = smem_u32(smem) + warp * (D * TILE_BYTES);
  const uint32_t bar0 = smem_u32(smem) + WARPS * D * TILE_BYTES + warp * (D * 8);

  const uint16_t* __restrict__ x = a.x + static_cast<int64_t>(shard) * a.shard_elems;
  uint8_t* shard_base = a.bundle + static_cast<size_t>(shard) * a.shard_bytes;
  uint8_t* __restrict__ codes = shard_base;
  float2* __restrict__ scales_out = reinterpret_cast<float2*>(shard_base + a.scales_off);

  const int64_t nblocks = a.nblocks;
  const WarpWork ww(nblocks, static_cast<int64_t>(blockIdx.x) * WARPS + warp,
                    static_cast<int64_t>(gridDim.x) * WARPS, BPT);
  const int count = ww.count;   // tiles of this warp

  if (lane == 0) {
    for (int s = 0; s < D; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();
  grid_launch_dependents();
  grid_dependency_wait();   // no global access before the preceding grid is done

  // Producer state, kept identical in every lane (lane 0 issues the copy):
  // next tile number `it` of this warp, its source and its stage.
  int it = 0, is = 0;
  auto issue_next = [&]() {
    if (lane == 0) {
      int64_t tb0;
      int tvb;
      ww.tile(it, tb0, tvb);
      const uint32_t bytes = static_cast<uint32_t>(tvb) * (NB * 2);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar0 + 8 * is, bytes);
      tma_load_1d(stage0 + is * TILE_BYTES, x + tb0 * NB, bytes, bar0 + 8 * is, policy);
    }
    ++it;
    is = (is + 1 == D) ? 0 : is + 1;
  };
  while (it < D && it < count) issue_next();

  float part_smax = 0.0f;   // header partials of this thread (lane j == 0 only)
  uint32_t part_cnt = 0;
  int k = 0, cs = 0;
  uint32_t cphase = 0;
  bool ok = true;

  // The tile being finished: its first block and blocks, stage, and this
  // lane's block's (alpha, s).
  int64_t b0 = 0;
  int vb = 0;
  uint32_t stage = 0;
  float alpha = 1.0f, sc = 1.0f;
  // Scale pair and header partials of the lane's block, the bulk store of the
  // tile's codes, and the refill of the previous tile's stage.
  auto finish_tile = [&]() {
    if (sub < vb && j == 0) {
      scales_out[b0 + sub] = make_float2(alpha, sc);     // 8 contiguous bytes per lane
      part_smax = fmaxf(part_smax, sc);
      part_cnt += (sc > 1.0f) ? 1u : 0u;
    }
    fence_proxy_async_smem();   // this lane's codes are visible to the bulk store
    __syncwarp();
    if (lane == 0) {
      tma_store_1d(codes + b0 * NB, stage, static_cast<uint32_t>(vb) * NB);
      bulk_commit();
    }
    // Refill the stage of the previous tile once its codes have left it.
    if (k >= 1 && it < count) {
      if (lane == 0) bulk_wait_read<1>();
      issue_next();
    }
  };

  while (k < count) {
    // The common path, tile after tile. A tile with a non-zero block whose
    // sum of squares is not a trusted fp32 number (values far below or above
    // 1) leaves the loop unfinished and is redone below with each such block
    // scaled by a power of two (far_tile); keeping that call out of this loop
    // keeps the loop's code what it is without it.
    bool redo = false;
    float tmax_far = 0.0f;
    bool far = false;
    for (; k < count; ++k) {
      const bool got = mbar_wait(bar0 + 8 * cs, cphase);
      if (!__all_sync(kFullMask, got)) {   // keep the warp's decision uniform
        ok = false;
        break;
      }
      ww.tile(k, b0, vb);
      stage = stage0 + cs * TILE_BYTES;

      f2 v[kCH][4];
      {
        const uint32_t base = stage + sub * (NB * 2);
#pragma unroll
        for (int q = 0; q < kCH; ++q) {
          const uint4 r = lds128(base + 16 * (j + LPB * (q ^ cx)));
          v[q][0] = f2{bf16_lo(r.x), bf16_hi(r.x)};
          v[q][1] = f2{bf16_lo(r.y), bf16_hi(r.y)};
          v[q][2] = f2{bf16_lo(r.z), bf16_hi(r.z)};
          v[q][3] = f2{bf16_lo(r.w), bf16_hi(r.w)};
        }
      }
      if (++cs == D) {
        cs = 0;
        cphase ^= 1u;
      }

      // Block energy e = sum x^2 (E = e / NB): four packed accumulators, then
      // the lanes of the block.
      f2 ea[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int q = 0; q < kCH; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i) ea[i] = fma2(v[q][i], v[q][i], ea[i]);
      const f2 e01 = add2(ea[0], ea[1]), e23 = add2(ea[2], ea[3]);
      const float e = block_sum<LPB>((e01.x + e01.y) + (e23.x + e23.y));

      // alpha = sqrt(E*/E) = sqrt(n E*) / sqrt(e): reciprocal square root
      // with one Newton step (error about one ulp), kept in [2^-126, 2^126];
      // 1 for an all-zero block. It does not depend on the rotation, so its
      // latency overlaps the FWHT.
      float r = rsqrtf(e);
      r = fmaf(fmaf(-0.5f * e * r, r, 0.5f), r, r);
      alpha = (e > 0.f) ? clamp_alpha(a.sqrt_nE * r) : 1.0f;
      const float cscale = alpha * a.inv_sqrt_n;      // y = cscale * t

      // Rotation of the raw block: t = H x.
      fwht_in_registers<kCH>(v, cx);
      fwht_across_lanes<kCH, LPB>(v, j);

      // max |t| = max(max t, -min t): a tree of 3-input max / min per chunk,
      // then over the chunks.
      float hq[kCH], lq[kCH];
#pragma unroll
      for (int q = 0; q < kCH; ++q) {
        hq[q] = max3(max3(v[q][0].x, v[q][0].y, v[q][1].x), max3(v[q][1].y, v[q][2].x, v[q][2].y),
                     fmaxf(v[q][3].x, v[q][3].y));
        lq[q] = min3(min3(v[q][0].x, v[q][0].y, v[q][1].x), min3(v[q][1].y, v[q][2].x, v[q][2].y),
                     fminf(v[q][3].x, v[q][3].y));
      }
      const float thi = max3(max3(hq[0], hq[1], hq[2]), max3(hq[3], hq[4], hq[5]), fmaxf(hq[6], hq[7]));
      const float tlo = min3(min3(lq[0], lq[1], lq[2]), min3(lq[3], lq[4], lq[5]), fminf(lq[6], lq[7]));
      const float tmax = block_max<LPB>(fmaxf(thi, -tlo));

      const float amax = cscale * tmax;
      sc = (VARIANT == 0)   ? fmaxf(1.0f, amax * (1.0f / 448.0f))
           : (VARIANT == 1) ? (amax > 0.f ? amax * (1.0f / 448.0f) : 1.0f)
                            : a.s_static;
      const float g = __fdividef(cscale, sc);         // code value = g * t
      const f2 g2{g, g};

      // Codes go back into the stage this tile came from (the tile's codes
      // are half its bytes), then leave as one bulk store.
      __syncwarp();   // every lane has read the stage before any lane overwrites it
      {
        const uint32_t base = stage + sub * NB;
#pragma unroll
        for (int q = 0; q < kCH; ++q) {
          const f2 y0 = mul2(v[q][0], g2), y1 = mul2(v[q][1], g2);
          const f2 y2 = mul2(v[q][2], g2), y3 = mul2(v[q][3], g2);
          uint2 w;
          w.x = e4m3x4_from_f32(y0.x, y0.y, y1.x, y1.y);
          w.y = e4m3x4_from_f32(y2.x, y2.y, y3.x, y3.y);
          sts64(base + 8 * (j + LPB * (q ^ cx)), w);
        }
      }
      far = !(e >= kEnergyLo && e <= kEnergyHi) && !(tmax == 0.f);
      if (__any_sync(kFullMask, far)) {
        tmax_far = tmax;
        redo = true;
        break;
      }
      finish_tile();
    }
    if (!redo) break;
    // max |x| <= max |t| <= n max |x|: the scaled block's max lies in [2^-8, 2)
    const int kf = far ? (tmax_far <= 0x1.fffffep127f ? ilogbf(tmax_far) : 128) : 0;
    const float2 as = far_tile<NB, VARIANT>(x + b0 * NB, sub < vb, stage, sub, j, cx, kf, a.sqrt_nE,
                                            a.inv_sqrt_n, a.s_static);
    alpha = as.x;
    sc = as.y;
    finish_tile();
    ++k;
  }

  if (!ok) {
    // A stage never completed: record it, then wait (bounded) for the copies
    // this warp still has in flight (tiles k .. it-1) before the CTA may exit.
    if (lane == 0) atomicOr(&g_compress_fault, kFaultCompressWait);
    for (int kk = k; kk < it; ++kk) {
      mbar_wait(bar0 + 8 * cs, cphase);
      if (++cs == D) {
        cs = 0;
        cphase ^= 1u;
      }
    }
  }
  // ---- per-tensor header: CTA reduction, then the last CTA of the shard ----
  finish_header<kCompressThreads>(part_smax, part_cnt, a.workspace + shard * kWorkspaceShardStride,
                                  a.headers + shard, a.N, a.h, NB, VARIANT, a.target_energy, a.q_max);
  // the stages may be released once every store has read them (the kernel's
  // end makes the stored codes visible)
  if (lane == 0) bulk_wait_read<0>();
}

template <int NB>
void (*kernel_fn(int variant))(CompressArgs) {
  return variant == 0 ? compress_kernel<NB, 0> : variant == 1 ? compress_kernel<NB, 1> : compress_kernel<NB, 2>;
}

}  // namespace

size_t compress_smem_bytes() {
  return static_cast<size_t>(kCompressThreads / 32) * kCompressStages * (kTileElems * 2 + 8);
}

const void* compress_kernel_ptr(int block, int variant) {
  switch (block) {
    case 64: return reinterpret_cast<const void*>(kernel_fn<64>(variant));
    case 128: return reinterpret_cast<const void*>(kernel_fn<128>(variant));
    default: return reinterpret_cast<const void*>(kernel_fn<256>(variant));
  }
}

cudaError_t launch_compress(const CompressArgs& a, int block, int variant, int grid_x, int P,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, P);
  cfg.blockDim = dim3(kCompressThreads);
  cfg.dynamicSmemBytes = compress_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void (*kern)(CompressArgs) = block == 64    ? kernel_fn<64>(variant)
                               : block == 128 ? kernel_fn<128>(variant)
                                              : kernel_fn<256>(variant);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t compress_fault(unsigned int* bits, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_compress_fault, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_compress_fault, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace taco

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
// One CTA of 16 warps per SM. Each warp walks warp tiles (2048 elements) in
// grid-stride rounds and then an even share of the blocks left over
// (WarpWork); with CLAIM (E4M3 decompress-reduce, at least kClaimRounds full
// rounds per warp) the warps of a CTA claim the same tiles in order instead
// (CtaWork). For one tile a warp consumes P stages, one per shard; lane 0 keeps
// kDecompressStages stages in flight, each a pair of 1-D cp.async.bulk
// copies (the tile's codes and its (alpha, s) pairs) completed on one mbarrier.
// Codes are decoded in pairs with cvt.rn.f16x2.e4m3x2 (FMT 0) or, for the
// INT8 fallback format (FMT 1, pt summary §5), by placing the byte under a
// fixed exponent, and accumulated with packed f32x2 FMAs; the bf16 output
// tile is assembled in shared memory and leaves as one TMA bulk store.

#include "taco_device.cuh"
#include "taco_launch.h"

namespace taco {

namespace {

__device__ unsigned int g_decompress_fault;

constexpr uint32_t kCodesBytes = kTileElems;          // codes of one tile
constexpr uint32_t kScaleBytes = 256;                 // (alpha, s) pairs of one tile
constexpr uint32_t kStageBytes = kCodesBytes + kScaleBytes;
constexpr uint32_t kOutBytes = kTileElems * 2;        // bf16 output of one tile

// MODE 0: decompress-reduce to bf16.
// MODE 2: decompress without a sum: shard blockIdx.y to output rows
//         blockIdx.y * N .. (the AllGather side of the two-shot AllReduce).
// MODE 1: reduce-recompress. The sum x_hat = H z of the P reconstructions is
// compressed again without leaving the rotated domain: H x_hat = n z and
// sum x_hat^2 = n sum z^2 (H symmetric, H H = n I), so alpha' = sqrt(E* /
// sum z^2), the rotated block is alpha' sqrt(n) z and no transform is
// needed; the bf16 sum is written too when `out` is not null. gridDim.y
// independent reductions run in one launch: reduction y takes shards
// y*P .. y*P+P-1 and writes shard y, header y and workspace y.
// Four codes of one 32-bit word -> (elements 0, 1), (elements 2, 3).
template <int FMT>
__device__ __forceinline__ void decode4(uint32_t w, f2& v01, f2& v23) {
  if constexpr (FMT == 0) {
    v01 = e4m3x2_to_f2(w & 0xffffu);
    v23 = e4m3x2_to_f2(w >> 16);
  } else {
    i8x4_to_f32(w, v01, v23);
  }
}

template <int NB, int MODE, int VARIANT, int FMT = 0, bool CLAIM = false>
__global__ void __launch_bounds__(kDecompressThreads, kDecompressMinBlocks)
decompress_reduce_kernel(DecompressArgs a) {
  constexpr int LPB = NB / 64;
  constexpr int BPT = 32 / LPB;
  // Stages in flight per warp: 3 for the n = 128 decompress-reduce of E4M3
  // codes, 4 for the other shapes, modes and formats (measured on GB300:
  // qwen-7b-long 96.2 -> 93.8 us and gpt3-6.7b-act 57.1 -> 56.0 us with 3;
  // the reduce-recompress at n = 128, the INT8 codes (95.9 -> 96.9 us) and
  // every launch at n = 256 were as fast or faster with 4, and 2 was slower
  // everywhere). The shared memory is sized for 4.
  constexpr int D = (NB == 128 && MODE == 0 && FMT == 0) ? 3 : kDecompressStages;
  constexpr int WARPS = kDecompressThreads / 32;
  static_assert(LPB >= 1 && LPB <= 4, "block size");
  static_assert(BPT * 8 <= kScaleBytes, "scale slot");
  static_assert(D <= kDecompressStages, "the shared memory holds kDecompressStages stages per warp");

  extern __shared__ __align__(128) unsigned char smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = lane & (LPB - 1);
  const int sub = lane / LPB;
  const int cx = sub & (kCH - 1);
  const int P = (MODE == 2) ? 1 : a.P;
  const uint8_t* const* shard_of = (MODE == 2)   ? a.shard + blockIdx.y
                                  : (MODE == 1) ? a.shard + blockIdx.y * a.P
                                                : a.shard;
  uint16_t* const out_base = (MODE == 2) ? a.out + static_cast<int64_t>(blockIdx.y) * a.nblocks * NB : a.out;
  uint8_t* const rc_shard = (MODE == 1) ? a.rc_shard + blockIdx.y * a.rc_stride : nullptr;

  const uint32_t stage0 = smem_u32(smem) + warp * (D * kStageBytes);
  const uint32_t bar0 = smem_u32(smem) + WARPS * D * kStageBytes + warp * (D * 8);
  // this warp's output tile (bf16), written out with one bulk store per tile
  const uint32_t out0 = smem_u32(smem) + WARPS * D * (kStageBytes + 8) + warp * kOutBytes;

  const int64_t nblocks = a.nblocks;
  const WarpWork ww(nblocks, static_cast<int64_t>(blockIdx.x) * WARPS + warp,
                    static_cast<int64_t>(gridDim.x) * WARPS, BPT);
  const int ntiles = ww.count;
  const int count = ntiles * P;                       // stages of this warp
  // CLAIM: the CTA's warp tiles are a list (CtaWork) that its warps claim in
  // order instead of the fixed share above. When a warp's producer starts a
  // tile, lane 0 takes the next item from the shared counter and writes
  // (first block, blocks) into the warp's ring slot it_t & 3, or first
  // block -1 past the end; every lane reads the slot when the warp's
  // consumer starts that tile. The producer runs at most D - 1 stages ahead,
  // so a slot is read before it is written again.
  __shared__ int sh_next;
  const CtaWork cw(nblocks, blockIdx.x, gridDim.x, WARPS, BPT);
  const uint32_t ring0 = smem_u32(smem) + WARPS * D * (kStageBytes + 8) + WARPS * kOutBytes + warp * 64;

  if (CLAIM && threadIdx.x == 0) sh_next = 0;
  if (lane == 0) {
    for (int s = 0; s < D; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
  }
  if constexpr (CLAIM) {
    __syncthreads();
  } else {
    __syncwarp();
  }
  grid_launch_dependents();
  if (lane == 0) {
    // the first stages this warp copies (its first tile, or the CTA's item
    // with the warp's index, which the warps claim first; shards 0 .. D-1)
    // into L2 while the preceding grid finishes: a prefetch returns no
    // data, so it may come before the wait
    int64_t pb0 = -1;
    int pvb = 0;
    if constexpr (CLAIM) {
      if (!cw.item(warp, pb0, pvb)) pb0 = -1;
    } else if (ntiles > 0) {
      ww.tile(0, pb0, pvb);
    }
    if (pb0 >= 0 && pvb > 0)
      for (int p = 0; p < P && p < D; ++p) {
        bulk_prefetch_l2(shard_of[p] + pb0 * NB, static_cast<uint32_t>(pvb) * NB);
        bulk_prefetch_l2(shard_of[p] + a.scales_off + pb0 * 8, (static_cast<uint32_t>(pvb) * 8 + 15) & ~15u);
      }
  }
  grid_dependency_wait();   // no global access before the preceding grid is done

  // Producer state, kept identical in every lane (lane 0 issues the copies):
  // next stage = (tile number it_t of this warp, shard ip) and its slot is.
  // The reduce-recompress (MODE 1) keeps the tile's offsets, sizes and the
  // cache policy from the tile's first shard on: that removes its register
  // spills (n = 128, 256), while the other modes measured faster with them
  // recomputed for every stage.
  constexpr bool kKeepTile = (MODE == 1);
  int issued = 0, it_t = 0, ip = 0, is = 0;
  bool prod_done = false;   // CLAIM: the CTA's list is exhausted for this warp
  uint64_t k_policy = 0, k_codes = 0, k_scales = 0;   // kept tile (MODE 1)
  uint32_t k_cbytes = 0, k_sbytes = 0;
  if constexpr (kKeepTile) k_policy = l2_evict_first_policy();
  auto issue_next = [&]() {
    if constexpr (CLAIM) {
      if (ip == 0) {
        // a new tile: claim it (lane 0); the warp follows lane 0's answer
        int got = 0;
        if (lane == 0) {
          int64_t tb0 = -1;
          int tvb = 0;
          got = cw.item(atomicAdd(&sh_next, 1), tb0, tvb) ? 1 : 0;
          if (!got) tb0 = -1;
          sts128(ring0 + 16 * (it_t & 3),
                 make_uint4(static_cast<uint32_t>(tb0), static_cast<uint32_t>(static_cast<uint64_t>(tb0) >> 32),
                            static_cast<uint32_t>(tvb), 0u));
        }
        if (!__shfl_sync(kFullMask, got, 0)) {
          prod_done = true;
          return;
        }
      }
    }
    if (lane == 0) {
      uint64_t policy, off_codes, off_scales;
      uint32_t cbytes, sbytes;
      if (!kKeepTile || ip == 0) {
        int64_t tb0;
        int tvb;
        if constexpr (CLAIM) {
          const uint4 tr = lds128(ring0 + 16 * (it_t & 3));
          tb0 = static_cast<int64_t>((static_cast<uint64_t>(tr.y) << 32) | tr.x);
          tvb = static_cast<int>(tr.z);
        } else {
          ww.tile(it_t, tb0, tvb);
        }
        const uint32_t vb = static_cast<uint32_t>(tvb);
        off_codes = static_cast<uint64_t>(tb0) * NB;
        off_scales = a.scales_off + static_cast<uint64_t>(tb0) * 8;
        cbytes = vb * NB;
        sbytes = (vb * 8 + 15) & ~15u;   // stays inside the 256-byte padding
        if constexpr (kKeepTile) {
          k_codes = off_codes;
          k_scales = off_scales;
          k_cbytes = cbytes;
          k_sbytes = sbytes;
        }
      }
      if constexpr (kKeepTile) {
        policy = k_policy;
        off_codes = k_codes;
        off_scales = k_scales;
        cbytes = k_cbytes;
        sbytes = k_sbytes;
      } else {
        policy = l2_evict_first_policy();
      }
      const uint32_t dst = stage0 + is * kStageBytes;
      const uint32_t bar = bar0 + 8 * is;
      const uint8_t* base = shard_of[ip];
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, cbytes + sbytes);
      tma_load_1d(dst, base + off_codes, cbytes, bar, policy);
      tma_load_1d(dst + kCodesBytes, base + off_scales, sbytes, bar, policy);
    }
    ++issued;
    is = (is + 1 == D) ? 0 : is + 1;
    if (++ip == P) {
      ip = 0;
      ++it_t;
    }
  };
  auto more = [&]() { return CLAIM ? !prod_done : issued < count; };
  while (issued < D - 1 && more()) issue_next();
  if constexpr (CLAIM) __syncwarp();   // the ring slots lane 0 wrote are visible to the warp

  int k = 0, cs = 0;
  uint32_t cphase = 0;
  bool ok = true;
  float part_smax = 0.0f;   // reduce-recompress header partials (lane j == 0)
  uint32_t part_cnt = 0;
  for (int ti = 0; (CLAIM || ti < ntiles) && ok; ++ti) {
    int64_t b0;   // first block of the tile
    int vb;       // blocks in the tile
    if constexpr (CLAIM) {
      const uint4 tr = lds128(ring0 + 16 * (ti & 3));
      b0 = static_cast<int64_t>((static_cast<uint64_t>(tr.y) << 32) | tr.x);
      vb = static_cast<int>(tr.z);
      if (b0 < 0) break;   // the CTA's list is exhausted
    } else {
      ww.tile(ti, b0, vb);
    }

    f2 z[kCH][4];
#pragma unroll
    for (int q = 0; q < kCH; ++q)
#pragma unroll
      for (int i = 0; i < 4; ++i) z[q][i] = f2{0.f, 0.f};

    for (int p = 0; p < P; ++p, ++k) {
      if (more()) issue_next();
      const bool got = mbar_wait(bar0 + 8 * cs, cphase);
      if (!__all_sync(kFullMask, got)) {   // keep the warp's decision uniform
        ok = false;
        break;
      }
      const uint32_t st = stage0 + cs * kStageBytes;
      const uint2 as = lds64(st + kCodesBytes + 8 * sub);   // (alpha, s) of the block
      uint2 w[kCH];
#pragma unroll
      for (int q = 0; q < kCH; ++q) w[q] = lds64(st + sub * NB + 8 * (j + LPB * (q ^ cx)));
      __syncwarp();   // every lane has read slot cs: lane 0 may refill it
      if (++cs == D) {
        cs = 0;
        cphase ^= 1u;
      }

      // s / alpha / sqrt(n); alpha >= 2^-126 and < 2^126 for every finite
      // input the compress kernel accepts, inside __fdividef's range.
      const float d = __fdividef(__uint_as_float(as.y), __uint_as_float(as.x)) * a.inv_sqrt_n;
      const f2 d2{d, d};
#pragma unroll
      for (int q = 0; q < kCH; ++q) {
        f2 c0, c1, c2, c3;
        decode4<FMT>(w[q].x, c0, c1);
        decode4<FMT>(w[q].y, c2, c3);
        z[q][0] = fma2(d2, c0, z[q][0]);
        z[q][1] = fma2(d2, c1, z[q][1]);
        z[q][2] = fma2(d2, c2, z[q][2]);
        z[q][3] = fma2(d2, c3, z[q][3]);
      }
    }
    if (!ok) break;

    if constexpr (MODE == 1) {
      // energy of x_hat: sum x_hat^2 / n = sum z^2, summed in an order that
      // does not depend on the block's place in the tile
      const float e = block_sum<LPB>(lane_sum_squares<false>(z, f2{1.f, 1.f}, f2{1.f, 1.f}));
      float r = rsqrtf(e);
      r = fmaf(fmaf(-0.5f * e * r, r, 0.5f), r, r);
      float alpha = (e > 0.f) ? clamp_alpha(a.sqrt_E * r) : 1.0f;   // kept in [2^-126, 2^126]
      float hq[kCH], lq[kCH];
#pragma unroll
      for (int q = 0; q < kCH; ++q) {
        hq[q] = max3(max3(z[q][0].x, z[q][0].y, z[q][1].x), max3(z[q][1].y, z[q][2].x, z[q][2].y),
                     fmaxf(z[q][3].x, z[q][3].y));
        lq[q] = min3(min3(z[q][0].x, z[q][0].y, z[q][1].x), min3(z[q][1].y, z[q][2].x, z[q][2].y),
                     fminf(z[q][3].x, z[q][3].y));
      }
      const float zhi = max3(max3(hq[0], hq[1], hq[2]), max3(hq[3], hq[4], hq[5]), fmaxf(hq[6], hq[7]));
      const float zlo = min3(min3(lq[0], lq[1], lq[2]), min3(lq[3], lq[4], lq[5]), fminf(lq[6], lq[7]));
      const float zmax = block_max<LPB>(fmaxf(zhi, -zlo));
      // A non-zero block whose sum of squares is not a trusted fp32 number:
      // its energy is taken again from 2^-k z (k the exponent of max |z|;
      // exact) and 2^-k is put back into alpha. z itself is not changed, and
      // blocks that are not far take k = 0 and repeat the arithmetic above.
      const bool far = !(e >= kEnergyLo && e <= kEnergyHi) && !(zmax == 0.f);
      const bool any_far = __any_sync(kFullMask, far);
      const int k = (far && zmax <= 0x1.fffffep127f) ? ilogbf(zmax) : 0;
      const int nk = -k, nk1 = nk >> 1;              // 2^-k = 2^nk1 2^(nk - nk1), both normal
      const f2 s1{exp2i(nk1), exp2i(nk1)}, s2{exp2i(nk - nk1), exp2i(nk - nk1)};
      if (any_far) {
        const float e2 = block_sum<LPB>(lane_sum_squares<true>(z, s1, s2));
        float r2 = rsqrtf(e2);
        r2 = fmaf(fmaf(-0.5f * e2 * r2, r2, 0.5f), r2, r2);
        alpha = (e2 > 0.f) ? clamp_alpha(a.sqrt_E * r2 * s1.x * s2.x) : 1.0f;
      }
      // rotated block = alpha sqrt(n) z; a far block takes its codes from
      // 2^-k z with alpha 2^k sqrt(n), which stays in the fp32 range where
      // alpha sqrt(n) or y / s would not (k = 0 elsewhere: no change)
      const float cscale = ldexpf(alpha, k) * a.sqrt_n;
      const float amax = cscale * ldexpf(zmax, -k);
      constexpr float QMAX = (FMT == 0) ? 448.0f : 127.0f;
      const float sc = (VARIANT == 0)   ? fmaxf(1.0f, amax * (1.0f / QMAX))
                       : (VARIANT == 1) ? (amax > 0.f ? amax * (1.0f / QMAX) : 1.0f)
                                        : a.s_static;
      const float g = __fdividef(cscale, sc);
      const f2 g2{g, g};
      if (lane == 0) bulk_wait_read<0>();   // the previous store has read the buffer
      __syncwarp();
      if (any_far)
        store_codes<FMT, LPB, true, VARIANT == 2>(z, g2, s1, s2, out0 + sub * NB, j, cx);
      else
        store_codes<FMT, LPB, false, VARIANT == 2>(z, g2, s1, s2, out0 + sub * NB, j, cx);
      if (sub < vb && j == 0) {
        reinterpret_cast<float2*>(rc_shard + a.scales_off)[b0 + sub] = make_float2(alpha, sc);
        part_smax = fmaxf(part_smax, sc);
        part_cnt += (sc > 1.0f) ? 1u : 0u;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_1d(rc_shard + b0 * NB, out0, static_cast<uint32_t>(vb) * NB);
        bulk_commit();
      }
      if (a.out == nullptr) continue;
    }

    fwht_in_registers<kCH>(z, cx);
    fwht_across_lanes<kCH, LPB>(z, j);

    // Output tile through shared memory and one bulk store (contiguous).
    if (lane == 0) bulk_wait_read<0>();   // the previous tile's store has read the buffer
    __syncwarp();
    {
      const uint32_t base = out0 + sub * (NB * 2);
#pragma unroll
      for (int q = 0; q < kCH; ++q) {
        uint4 o;
        o.x = pack_bf16x2(z[q][0].x, z[q][0].y);
        o.y = pack_bf16x2(z[q][1].x, z[q][1].y);
        o.z = pack_bf16x2(z[q][2].x, z[q][2].y);
        o.w = pack_bf16x2(z[q][3].x, z[q][3].y);
        sts128(base + 16 * (j + LPB * (q ^ cx)), o);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_1d(out_base + b0 * NB, out0, static_cast<uint32_t>(vb) * (NB * 2));
      bulk_commit();
    }
  }

  if (!ok) {
    // A stage never completed: record it, then wait (bounded) for the copies
    // this warp still has in flight (stages k .. issued-1) before it exits.
    if (lane == 0) atomicOr(&g_decompress_fault, kFaultDecompressWait);
    for (int kk = k; kk < issued; ++kk) {
      mbar_wait(bar0 + 8 * cs, cphase);
      if (++cs == D) {
        cs = 0;
        cphase ^= 1u;
      }
    }
  }
  if constexpr (MODE == 1) {
    finish_header<kDecompressThreads>(part_smax, part_cnt, a.workspace + blockIdx.y * kWorkspaceShardStride,
                                      a.rc_header + blockIdx.y, a.N, a.h, NB,
                                      VARIANT, a.target_energy, FMT == 0 ? 448.0f : 127.0f);
  }
  // the buffers may be released once every store has read them (the
  // kernel's end makes the stored output visible)
  if (lane == 0) bulk_wait_read<0>();
}

}  // namespace

size_t decompress_smem_bytes() {
  // per warp: stages, their barriers, the output tile and the 4-slot tile ring
  return static_cast<size_t>(kDecompressThreads / 32) *
         (kDecompressStages * (kStageBytes + 8) + kOutBytes + 64);
}

namespace {
template <int FMT, bool CLAIM>
void (*decompress_fn_claim(int block))(DecompressArgs) {
  return block == 64    ? decompress_reduce_kernel<64, 0, 0, FMT, CLAIM>
         : block == 128 ? decompress_reduce_kernel<128, 0, 0, FMT, CLAIM>
                        : decompress_reduce_kernel<256, 0, 0, FMT, CLAIM>;
}
void (*decompress_fn(int block, int fmt, bool claim))(DecompressArgs) {
  return fmt == 0 ? (claim ? decompress_fn_claim<0, true>(block) : decompress_fn_claim<0, false>(block))
                  : (claim ? decompress_fn_claim<1, true>(block) : decompress_fn_claim<1, false>(block));
}
}  // namespace

const void* decompress_kernel_ptr(int block, int fmt, bool claim) {
  return reinterpret_cast<const void*>(decompress_fn(block, fmt, claim));
}

namespace {
template <int NB, int FMT, bool CLAIM>
void (*recompress_fn_fmt(int variant))(DecompressArgs) {
  return variant == 0   ? decompress_reduce_kernel<NB, 1, 0, FMT, CLAIM>
         : variant == 1 ? decompress_reduce_kernel<NB, 1, 1, FMT, CLAIM>
                        : decompress_reduce_kernel<NB, 1, 2, FMT, CLAIM>;
}
// claim: the warps of a CTA claim its tiles in order (E4M3 codes only)
template <int NB>
void (*recompress_fn(int variant, int fmt, bool claim = false))(DecompressArgs) {
  return fmt != 0 ? recompress_fn_fmt<NB, 1, false>(variant)
         : claim  ? recompress_fn_fmt<NB, 0, true>(variant)
                  : recompress_fn_fmt<NB, 0, false>(variant);
}
template <int NB>
void (*gather_fn(int fmt))(DecompressArgs) {
  return fmt == 0 ? decompress_reduce_kernel<NB, 2, 0, 0> : decompress_reduce_kernel<NB, 2, 0, 1>;
}
}  // namespace

const void* recompress_kernel_ptr(int block, int variant, int fmt, bool claim) {
  switch (block) {
    case 64: return reinterpret_cast<const void*>(recompress_fn<64>(variant, fmt, claim));
    case 128: return reinterpret_cast<const void*>(recompress_fn<128>(variant, fmt, claim));
    default: return reinterpret_cast<const void*>(recompress_fn<256>(variant, fmt, claim));
  }
}

cudaError_t launch_decompress(const DecompressArgs& a, int block, int fmt, int grid,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecompressThreads);
  cfg.dynamicSmemBytes = decompress_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // With E4M3 codes, warps with at least kClaimRounds full grid-stride
  // rounds claim their CTA's tiles in order (the warps the scheduler favours
  // take more): 2-2.6% faster on the large tensors measured. With fewer
  // rounds, and for the INT8 codes (2% slower claimed on gpt3-act), the fixed
  // share per warp measured faster.
  const int64_t bpt = 32 / (block / 64);
  const int64_t rounds = a.nblocks / (static_cast<int64_t>(grid) * (kDecompressThreads / 32) * bpt);
  void (*kern)(DecompressArgs) = decompress_fn(block, fmt, fmt == 0 && rounds >= kClaimRounds);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_decompress_shards(const DecompressArgs& a, int block, int fmt, int grid, int P,
                                     cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, P);
  cfg.blockDim = dim3(kDecompressThreads);
  cfg.dynamicSmemBytes = decompress_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void (*kern)(DecompressArgs) = block == 64    ? gather_fn<64>(fmt)
                                 : block == 128 ? gather_fn<128>(fmt)
                                                : gather_fn<256>(fmt);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

const void* gather_kernel_ptr(int block, int fmt) {
  switch (block) {
    case 64: return reinterpret_cast<const void*>(gather_fn<64>(fmt));
    case 128: return reinterpret_cast<const void*>(gather_fn<128>(fmt));
    default: return reinterpret_cast<const void*>(gather_fn<256>(fmt));
  }
}

cudaError_t launch_reduce_recompress(const DecompressArgs& a, int block, int variant, int fmt,
                                     int grid, int batch, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, batch);
  cfg.blockDim = dim3(kDecompressThreads);
  cfg.dynamicSmemBytes = decompress_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // With E4M3 codes and at least kClaimRounds full grid-stride rounds per
  // warp, the warps claim their CTA's tiles in order, as the
  // decompress-reduce does: measured gpt3-6.7b-act 53.0 -> 52.2 us,
  // gpt3-6.7b-grad 52.2 -> 51.9, qwen-7b-long 87.9 -> 86.6.
  const int64_t bpt = 32 / (block / 64);
  const int64_t rounds = a.nblocks / (static_cast<int64_t>(grid) * (kDecompressThreads / 32) * bpt);
  const bool claim = fmt == 0 && rounds >= kClaimRounds;
  void (*kern)(DecompressArgs) = block == 64    ? recompress_fn<64>(variant, fmt, claim)
                                 : block == 128 ? recompress_fn<128>(variant, fmt, claim)
                                                : recompress_fn<256>(variant, fmt, claim);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t decompress_fault(unsigned int* bits, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_decompress_fault, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_decompress_fault, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace taco

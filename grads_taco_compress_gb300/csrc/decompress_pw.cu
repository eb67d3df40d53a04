// Decompress-reduce and reduce-recompress with a producer warp, for every
// block size and both code formats.
//
// The arithmetic is the one of decompress_reduce.cu ("TACO: Efficient
// Communication Compression of Intermediate Tensors ...", gist.science pt
// summary, §2.B.2 reconstruction with the two scales, §2.B.3 the reduce of
// the ReduceScatter half of the two-shot AllReduce and the recompression of
// the reduced chunk for the AllGather):
//   z      = sum_p (s_p / alpha_p / sqrt(n)) dec(q_p)     (fp32, rotated domain)
//   x_hat  = bf16( H_n z )                                 (MODE 0, and MODE 1's side output)
//   MODE 1 also compresses x_hat again without leaving the rotated domain:
//   alpha' = sqrt(E* / sum z^2), rotated block = alpha' sqrt(n) z.
// Every lane keeps the per-element layout of that file (a block spans
// LPB = n / 64 lanes, 8 chunks of 8 elements per lane, chunk slots XORed by
// the block's index in the warp tile), so the outputs are the same bits.
//
// What differs is who moves the data. One CTA of 16 warps per SM: warp 15
// alone issues the copies, one shard of a CTA tile per stage (the tile's
// codes and its (alpha, s) pairs, two 1-D bulk copies), into a ring of
// kStages stages that the 15 consumer warps share. A CTA tile is 15 warp
// tiles of 2048 elements (480, 240 or 120 blocks); consumer warp w reads warp
// tile w of every stage and arrives on the stage's "empty" barrier once it
// has read it, so the consumers spend no issue slots on copy bookkeeping.
// CTA tiles go in grid-stride rounds, then each CTA takes its even share of
// the blocks left over (4-block boundaries) in pieces of at most one tile.
// Every wait is bounded in time; a wait that gives up sets a CTA-wide abort
// flag and the kernel's fault bit, and the producer lets its copies in flight
// land before the CTA exits.

#include "taco_device.cuh"
#include "taco_launch.h"

namespace taco {

namespace {

__device__ unsigned int g_decompress_pw_fault;

constexpr int kPwCons = 15;                                  // consumer warps
constexpr uint32_t kPwCodes = kPwCons * kTileElems;          // codes of one CTA tile: 30720 B
static_assert(kPwCons + 1 == kDecompressThreads / 32, "one producer warp and the consumers");

template <int NB>
struct PwShape {
  static constexpr int LPB = NB / 64;                        // lanes per block
  static constexpr int BPT = 32 / LPB;                       // blocks per warp tile
  static constexpr int TB = kPwCons * BPT;                   // blocks per CTA tile
  static constexpr int kStages = 4;                          // stages in the ring
  static constexpr uint32_t stage = kPwCodes + TB * 8;       // codes + (alpha, s) pairs
  static constexpr uint32_t out = kTileElems * 2;            // per consumer warp: a bf16 warp tile
  // (reduce-recompress: the warp tile's codes, then its (alpha, s) pairs)
  static_assert(NB * BPT + 8 * BPT <= out, "codes and pairs of a warp tile fit the output buffer");
  static_assert((NB * BPT) % 16 == 0, "pairs staging 16-byte aligned");
  static constexpr uint32_t bars = kStages * stage + kPwCons * out;
  static constexpr uint32_t smem = bars + 2 * 8 * kStages + 16;
  static_assert(stage % 16 == 0 && out % 16 == 0, "TMA destinations 16-byte aligned");
};

// The CTA tiles of one CTA: full grid-stride rounds, then the CTA's even
// share of the blocks left over in pieces of at most TB blocks.
struct PwItems {
  int64_t G, c, tb, n_full, lo, hi, total;
  __device__ __forceinline__ PwItems(int64_t nblocks, int64_t c_, int64_t G_, int64_t tb_)
      : G(G_), c(c_), tb(tb_) {
    const int64_t rounds = nblocks / (G * tb);
    const int64_t rem0 = rounds * G * tb;
    const int64_t rest = nblocks - rem0;
    n_full = rounds;
    lo = rem0 + ((rest * c / G) & ~int64_t{3});
    hi = rem0 + ((c + 1 == G) ? rest : ((rest * (c + 1) / G) & ~int64_t{3}));
    if (hi < lo) hi = lo;
    total = n_full + (hi - lo + tb - 1) / tb;
  }
  // first block and number of blocks of the CTA's tile k (k < total)
  __device__ __forceinline__ void get(int64_t k, int64_t& b0, int& vb) const {
    if (k < n_full) {
      b0 = (k * G + c) * tb;
      vb = static_cast<int>(tb);
    } else {
      b0 = lo + (k - n_full) * tb;
      const int64_t left = hi - b0;
      vb = static_cast<int>(left < tb ? left : tb);
    }
  }
};

// bounded wait; gives up when the CTA's abort flag is set or after
// kWaitLimitNs, setting the flag and the kernel's fault bit
__device__ __forceinline__ bool pw_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1u;
      atomicOr(&g_decompress_pw_fault, kFaultDecompressWait);
      return false;
    }
  }
}

// Four codes of one 32-bit word -> (elements 0, 1), (elements 2, 3).
template <int FMT>
__device__ __forceinline__ void pw_decode4(uint32_t w, f2& v01, f2& v23) {
  if constexpr (FMT == 0) {
    v01 = e4m3x2_to_f2(w & 0xffffu);
    v23 = e4m3x2_to_f2(w >> 16);
  } else {
    i8x4_to_f32(w, v01, v23);
  }
}

// MODE 0: decompress-reduce of P shards into bf16 `out`.
// MODE 1: reduce-recompress; gridDim.y independent reductions, reduction y
// takes shards y*P .. y*P+P-1 and writes shard y, header y and workspace y;
// the bf16 sum too when `out` is not null (then gridDim.y == 1).
template <int NB, int MODE, int VARIANT, int FMT>
__global__ void __launch_bounds__(kDecompressThreads, 1) decompress_pw_kernel(DecompressArgs a) {
  using S = PwShape<NB>;
  constexpr int LPB = S::LPB, BPT = S::BPT, TB = S::TB;
  constexpr int kPwStages = S::kStages;
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t base = smem_u32(smem);
  const uint32_t full0 = base + S::bars, empty0 = full0 + 8 * kPwStages;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + S::bars + 16 * kPwStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.P;
  const uint8_t* const* shard_of = (MODE == 1) ? a.shard + blockIdx.y * a.P : a.shard;
  const PwItems it(a.nblocks, blockIdx.x, gridDim.x, TB);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPwStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kPwCons);
    }
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  grid_launch_dependents();
  if (warp == kPwCons && lane == 0) {
    // the CTA's first tile of the first shards (the first ring of stages)
    // into L2 while the preceding grid finishes (a prefetch returns no data,
    // so it may come before the wait)
    int64_t b0 = 0;
    int vb = 0;
    if (it.total > 0) it.get(0, b0, vb);
    if (vb > 0)
      for (int p = 0; p < P && p < kPwStages; ++p) {
        bulk_prefetch_l2(shard_of[p] + b0 * NB, static_cast<uint32_t>(vb) * NB);
        bulk_prefetch_l2(shard_of[p] + a.scales_off + b0 * 8, (static_cast<uint32_t>(vb) * 8 + 15) & ~15u);
      }
  }
  grid_dependency_wait();   // no global access before the preceding grid is done

  float part_smax = 0.0f;   // reduce-recompress header partials (lane j == 0)
  uint32_t part_cnt = 0;

  if (warp == kPwCons) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      uint32_t i = 0;
      bool ok = true;
      for (int64_t k = 0; k < it.total && ok; ++k) {
        int64_t b0;
        int vb;
        it.get(k, b0, vb);
        const uint32_t cbytes = static_cast<uint32_t>(vb) * NB;
        const uint32_t sbytes = (static_cast<uint32_t>(vb) * 8 + 15) & ~15u;   // inside the 256-byte padding
        for (int p = 0; p < P; ++p, ++i) {
          const uint32_t s = i % kPwStages, ph = (i / kPwStages) & 1u;
          if (!pw_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = base + s * S::stage;
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(full0 + 8 * s, cbytes + sbytes);
          tma_load_1d(dst, shard_of[p] + b0 * NB, cbytes, full0 + 8 * s, policy);
          tma_load_1d(dst + kPwCodes, shard_of[p] + a.scales_off + b0 * 8, sbytes, full0 + 8 * s, policy);
        }
      }
      // the copies in flight land before the CTA may exit
      const uint32_t first = i > static_cast<uint32_t>(kPwStages) ? i - kPwStages : 0u;
      for (uint32_t j = first; j < i; ++j) mbar_wait(full0 + 8 * (j % kPwStages), (j / kPwStages) & 1u);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers
    const int j = lane & (LPB - 1);          // lane inside its block
    const int sub = lane / LPB;              // block inside the warp tile
    const int cx = sub & (kCH - 1);          // chunk-slot swizzle
    const uint32_t out0 = base + kPwStages * S::stage + warp * S::out;
    const uint32_t wcodes = warp * kTileElems + sub * NB;   // this lane's block in a stage
    const uint32_t wscale = kPwCodes + 8 * (warp * BPT + sub);
    uint32_t i = 0;
    bool ok = true;
    for (int64_t k = 0; k < it.total && ok; ++k) {
      int64_t b0;
      int vb;
      it.get(k, b0, vb);
      int wvb = vb - BPT * warp;             // this warp's blocks of the tile
      wvb = wvb < 0 ? 0 : (wvb > BPT ? BPT : wvb);
      const int64_t wb0 = b0 + BPT * warp;   // first block of this warp's tile
      f2 z[kCH][4];
#pragma unroll
      for (int q = 0; q < kCH; ++q)
#pragma unroll
        for (int r = 0; r < 4; ++r) z[q][r] = f2{0.f, 0.f};
      for (int p = 0; p < P; ++p, ++i) {
        const uint32_t s = i % kPwStages, ph = (i / kPwStages) & 1u;
        const bool got = pw_wait(full0 + 8 * s, ph, abort_flag);
        if (!__all_sync(kFullMask, got)) {   // keep the warp's decision uniform
          ok = false;
          break;
        }
        const uint32_t st = base + s * S::stage;
        const uint2 as = lds64(st + wscale);                 // (alpha, s) of the block
        uint2 w[kCH];
#pragma unroll
        for (int q = 0; q < kCH; ++q) w[q] = lds64(st + wcodes + 8 * (j + LPB * (q ^ cx)));
        __syncwarp();   // every lane has read the stage: the warp releases it
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        // s / alpha / sqrt(n); alpha lies in [2^-126, 2^126], inside
        // __fdividef's range
        const float d = __fdividef(__uint_as_float(as.y), __uint_as_float(as.x)) * a.inv_sqrt_n;
        const f2 d2{d, d};
#pragma unroll
        for (int q = 0; q < kCH; ++q) {
          f2 c0, c1, c2, c3;
          pw_decode4<FMT>(w[q].x, c0, c1);
          pw_decode4<FMT>(w[q].y, c2, c3);
          z[q][0] = fma2(d2, c0, z[q][0]);
          z[q][1] = fma2(d2, c1, z[q][1]);
          z[q][2] = fma2(d2, c2, z[q][2]);
          z[q][3] = fma2(d2, c3, z[q][3]);
        }
      }
      if (!ok || wvb == 0) continue;

      if constexpr (MODE == 1) {
        // energy of x_hat: sum x_hat^2 / n = sum z^2, summed in an order that
        // does not depend on the block's place in the tile
        const float e = block_sum<LPB>(lane_sum_squares<false>(z, f2{1.f, 1.f}, f2{1.f, 1.f}));
        float rr = rsqrtf(e);
        rr = fmaf(fmaf(-0.5f * e * rr, rr, 0.5f), rr, rr);
        float alpha = (e > 0.f) ? clamp_alpha(a.sqrt_E * rr) : 1.0f;   // kept in [2^-126, 2^126]
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
        // exact) and 2^-k is put back into alpha; z itself is not changed.
        const bool far = !(e >= kEnergyLo && e <= kEnergyHi) && !(zmax == 0.f);
        const bool any_far = __any_sync(kFullMask, far);
        const int kx = (far && zmax <= 0x1.fffffep127f) ? ilogbf(zmax) : 0;
        const int nk = -kx, nk1 = nk >> 1;           // 2^-k = 2^nk1 2^(nk - nk1), both normal
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
        const float cscale = ldexpf(alpha, kx) * a.sqrt_n;
        const float amax = cscale * ldexpf(zmax, -kx);
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
        // the (alpha, s) pairs are staged after the codes and stored by the
        // copy engine too: no plain global stores stay in flight, so the
        // release that publishes the header share waits for none
        uint8_t* const rc_shard = a.rc_shard + blockIdx.y * a.rc_stride;
        float2* const pairs_out = reinterpret_cast<float2*>(rc_shard + a.scales_off) + wb0;
        const uint32_t pstage = out0 + NB * BPT;
        if (j == 0) sts64(pstage + 8 * sub, make_uint2(__float_as_uint(alpha), __float_as_uint(sc)));
        if (sub < wvb && j == 0) {
          part_smax = fmaxf(part_smax, sc);
          part_cnt += (sc > 1.0f) ? 1u : 0u;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_1d(rc_shard + wb0 * NB, out0, static_cast<uint32_t>(wvb) * NB);
          // whole 16-byte pairs of blocks (wb0 is even); an odd last block
          // goes out from its lane
          if (wvb >= 2) tma_store_1d(pairs_out, pstage, static_cast<uint32_t>(wvb & ~1) * 8);
          bulk_commit();
        }
        if ((wvb & 1) && sub == wvb - 1 && j == 0) pairs_out[sub] = make_float2(alpha, sc);
        if (a.out == nullptr) continue;
      }

      fwht_in_registers<kCH>(z, cx);
      fwht_across_lanes<kCH, LPB>(z, j);
      if (lane == 0) bulk_wait_read<0>();   // the previous store has read the buffer
      __syncwarp();
      {
        const uint32_t ob = out0 + sub * (NB * 2);
#pragma unroll
        for (int q = 0; q < kCH; ++q) {
          uint4 o;
          o.x = pack_bf16x2(z[q][0].x, z[q][0].y);
          o.y = pack_bf16x2(z[q][1].x, z[q][1].y);
          o.z = pack_bf16x2(z[q][2].x, z[q][2].y);
          o.w = pack_bf16x2(z[q][3].x, z[q][3].y);
          sts128(ob + 16 * (j + LPB * (q ^ cx)), o);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_1d(a.out + wb0 * NB, out0, static_cast<uint32_t>(wvb) * (NB * 2));
        bulk_commit();
      }
    }
  }
  if constexpr (MODE == 1) {
    finish_header<kDecompressThreads>(part_smax, part_cnt, a.workspace + blockIdx.y * kWorkspaceShardStride,
                                      a.rc_header + blockIdx.y, a.N, a.h, NB, VARIANT, a.target_energy,
                                      FMT == 0 ? 448.0f : 127.0f);
  }
  // the buffers may be released once every store has read them (the
  // kernel's end makes the stored outputs visible)
  if (lane == 0) bulk_wait_read<0>();
}

template <int NB, int MODE, int FMT>
void (*pw_fn_v(int variant))(DecompressArgs) {
  if constexpr (MODE == 0) {
    return decompress_pw_kernel<NB, 0, 0, FMT>;
  } else {
    return variant == 0   ? decompress_pw_kernel<NB, 1, 0, FMT>
           : variant == 1 ? decompress_pw_kernel<NB, 1, 1, FMT>
                          : decompress_pw_kernel<NB, 1, 2, FMT>;
  }
}

template <int MODE>
void (*pw_fn(int block, int variant, int fmt))(DecompressArgs) {
  if (fmt == 0)
    return block == 64 ? pw_fn_v<64, MODE, 0>(variant)
                       : (block == 128 ? pw_fn_v<128, MODE, 0>(variant) : pw_fn_v<256, MODE, 0>(variant));
  return block == 64 ? pw_fn_v<64, MODE, 1>(variant)
                     : (block == 128 ? pw_fn_v<128, MODE, 1>(variant) : pw_fn_v<256, MODE, 1>(variant));
}

void (*pw_kernel(int mode, int block, int variant, int fmt))(DecompressArgs) {
  return mode == 0 ? pw_fn<0>(block, variant, fmt) : pw_fn<1>(block, variant, fmt);
}

}  // namespace

size_t decompress_pw_smem_bytes(int block) {
  return block == 64 ? PwShape<64>::smem : (block == 128 ? PwShape<128>::smem : PwShape<256>::smem);
}

int64_t decompress_pw_tile_blocks(int block) {
  return block == 64 ? PwShape<64>::TB : (block == 128 ? PwShape<128>::TB : PwShape<256>::TB);
}

const void* decompress_pw_kernel_ptr(int mode, int block, int variant, int fmt) {
  return reinterpret_cast<const void*>(pw_kernel(mode, block, variant, fmt));
}

cudaError_t launch_decompress_pw(const DecompressArgs& a, int mode, int block, int variant, int fmt,
                                 int grid, int batch, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, batch);
  cfg.blockDim = dim3(kDecompressThreads);
  cfg.dynamicSmemBytes = decompress_pw_smem_bytes(block);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, pw_kernel(mode, block, variant, fmt), a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t decompress_pw_fault(unsigned int* bits, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_decompress_pw_fault, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_decompress_pw_fault, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace taco

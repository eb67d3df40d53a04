// TACO decompress-reduce with the inverse rotation on the tensor cores
// (tcgen05, E4M3 operands), an alternative to decompress_reduce.cu with the
// same output.
//
// The reconstruction of the pt summary (§2.B.2), fused with the reduce of
// the ReduceScatter (§2.B.3):
//   x_hat = bf16( sum_p d_p H_n q_p ),   d_p = s_p / (alpha_p sqrt(n)),
// per block, q_p the decoded E4M3 codes of shard p. The rotation is linear,
// so each shard is rotated on its own and the scaled results are summed.
// With H_n = H_{n/64} (x) H_64 (Sylvester), u_{p,c} = H_64 q_{p,c} for every
// 64-code chunk c is one row of D = A_p * H_64^T on the tensor cores: A_p is
// the [128 blocks x 64] chunk of codes exactly as it arrives (kind::f8f6f4,
// E4M3), H_64 is +-1 in E4M3, and the fp32 accumulator holds u exactly (64
// products of E4M3 values by +-1 need at most 24 significant bits). The
// epilogue thread that owns a block sums d_p u_{p,c} over the shards and
// applies the remaining log2(n/64) butterfly levels across its chunks in
// registers, then writes bf16. No code is decoded on the CUDA cores.
//
// Shards are taken in groups of 256 / n, whose accumulators (n columns per
// shard) fill one of two 256-column halves of the tensor memory, so the
// MMAs of one half overlap the epilogue of the other. The sum of a block
// stays in registers (n fp32 values), which is why n = 256 is not offered.
//
// CTA = 10 warps, one CTA per SM (the two halves take all 512 TMEM columns;
// the shared memory does not fit twice):
//   warp 0     TMA producer: 2-D tensor loads of [128 blocks x 64 codes]
//              atoms (8 KB, 64-byte swizzle), shard by shard, chunk by chunk;
//   warp 1     owns the tensor memory; one lane issues 2 MMAs (K = 32) per
//              atom and commits each atom to its stage's "empty" barrier and
//              each shard group to the half's "full" barrier;
//   warps 2-9  two epilogue groups of 4 warps; group g takes the CTA's tiles
//              k with k % 2 == g from half g. Thread (warp w, lane l) owns
//              block row 32 (w % 4) + l. The (alpha, s) pairs are read from
//              global memory by the thread that needs them, ahead of the
//              wait. The bf16 tile leaves through 128-byte-swizzled TMA
//              tensor stores.
// Every wait is bounded in time with a CTA-wide abort flag, as in the
// tensor-core compress.

#include <cmath>

#include "taco_launch.h"
#include "tcgen05.cuh"

namespace taco {

namespace {

__device__ unsigned int g_decompress_mma_fault;

constexpr int kThreads = 320;
constexpr int kRows = 128;                            // blocks per tile (the MMA's M)
constexpr uint32_t kAtomBytes = kRows * 64;           // 8 KB of E4M3 codes
constexpr uint32_t kOutAtomBytes = kRows * 64 * 2;    // 16 KB of bf16
constexpr uint32_t kHBytes = 64 * 64;                 // H_64 in E4M3
constexpr uint32_t kTmemCols = 512;                   // two halves of 256
constexpr uint32_t kHalfCols = 256;
constexpr int kLoadCols = 32;                         // accumulator columns per tensor-memory wait

template <int NB>
struct DSmem {
  static constexpr int NC = NB / 64;
  static constexpr int GS = kHalfCols / NB;                         // shards per group
  static constexpr int kStages = NB == 64 ? 10 : 8;
  static constexpr uint32_t stages = 0;
  static constexpr uint32_t hmat = stages + kStages * kAtomBytes;
  static constexpr uint32_t out = hmat + kHBytes;                   // [group][chunk] atoms
  static constexpr uint32_t bars = out + 2 * NC * kOutAtomBytes;
  static constexpr uint32_t full = bars;
  static constexpr uint32_t empty = full + 8 * kStages;
  static constexpr uint32_t tfull = empty + 8 * kStages;
  static constexpr uint32_t tempty = tfull + 16;
  static constexpr uint32_t mma_done = tempty + 16;
  static constexpr uint32_t tmem_slot = mma_done + 8;
  static constexpr uint32_t abort_flag = tmem_slot + 4;
  static constexpr uint32_t end = abort_flag + 4;
  static constexpr uint32_t bytes = end + 1024;                     // + alignment slack
};

// One CTA per SM: a second one would wait for the tensor memory.
template <int NB>
constexpr bool one_cta_per_sm() {
  return DSmem<NB>::bytes <= 232448 && 233472 / (DSmem<NB>::bytes + 1024) == 1;
}
static_assert(one_cta_per_sm<64>() && one_cta_per_sm<128>(), "shared memory per CTA");

// E4M3 A and B, fp32 D, M = 128, N = 64.
constexpr uint32_t kIdesc = instr_desc(0, kRows, 64);

__device__ __forceinline__ uint64_t sw64_desc(uint32_t saddr) {
  return umma_desc(saddr, kSwizzle64, 512);   // 8 rows of 64 bytes per group
}

__device__ __forceinline__ bool wait_here(uint32_t bar, uint32_t parity,
                                          volatile uint32_t* abort_flag) {
  return wait_or_abort(bar, parity, abort_flag, &g_decompress_mma_fault, kFaultDecompressMmaWait);
}

struct DmmaMaps {
  CUtensorMap codes[TACO_MAX_SHARDS];   // shard p: [nblocks][n] bytes
  CUtensorMap out;                      // [nblocks][n] bf16
};

template <int NB>
__global__ void __launch_bounds__(kThreads, 1)
decompress_mma_kernel(const __grid_constant__ DmmaMaps maps, DecompressArgs a) {
  using S = DSmem<NB>;
  constexpr int NC = S::NC;
  constexpr int GS = S::GS;
  constexpr int kStages = S::kStages;

  extern __shared__ unsigned char smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem_raw + (base - smem_u32(smem_raw)) + S::abort_flag);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int P = a.P;
  const int ngroups = (P + GS - 1) / GS;
  const int64_t nblocks = a.nblocks;
  const int64_t ntiles = (nblocks + kRows - 1) / kRows;
  const int64_t G = gridDim.x;
  const int count = static_cast<int>(ntiles > blockIdx.x ? (ntiles - blockIdx.x + G - 1) / G : 0);

  // ---- set-up: barriers, H_64, tensor memory ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(base + S::full + 8 * s, 1);
      mbar_init(base + S::empty + 8 * s, 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(base + S::tfull + 8 * g, 1);
      mbar_init(base + S::tempty + 8 * g, 4);   // one arrival per epilogue warp
    }
    mbar_init(base + S::mma_done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  // H_64 as B in E4M3 (+1 = 0x38, -1 = 0xB8): 64 rows of 64 bytes, K-major,
  // 16-byte pieces swizzled by (row >> 1) & 3 (the 64-byte swizzle).
  for (int p = threadIdx.x; p < 64 * 4; p += kThreads) {
    const int r = p >> 2, piece = p & 3;
    uint32_t w[4];
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      uint32_t word = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int k = piece * 16 + k4 * 4 + b;
        word |= ((__popc(r & k) & 1) ? 0xB8u : 0x38u) << (8 * b);
      }
      w[k4] = word;
    }
    sts128(base + S::hmat + r * 64 + 16 * (piece ^ ((r >> 1) & 3)), make_uint4(w[0], w[1], w[2], w[3]));
  }
  fence_proxy_async_smem();   // H is read by the tensor cores (async proxy)
  if (warp == 1) tmem_alloc(base + S::tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds_u32(base + S::tmem_slot);

  grid_launch_dependents();
  grid_dependency_wait();   // no global access before the preceding grid is done

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer ----
    if (lane == 0) {
      for (int p = 0; p < P; ++p) prefetch_map(&maps.codes[p]);
      const uint64_t policy = l2_evict_first_policy();
      uint32_t i = 0;
      bool ok = true;
      for (int k = 0; k < count && ok; ++k) {
        const int row0 = static_cast<int>((blockIdx.x + k * G) * kRows);
        for (int p = 0; p < P && ok; ++p)
          for (int c = 0; c < NC; ++c, ++i) {
            const uint32_t s = i % kStages, ph = (i / kStages) & 1u;
            if (!wait_here(base + S::empty + 8 * s, ph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(base + S::full + 8 * s, kAtomBytes);
            tma_load_2d(base + S::stages + s * kAtomBytes, &maps.codes[p], c * 64, row0,
                        base + S::full + 8 * s, policy);
          }
      }
      if (!ok) {
        // copies still in flight land in their stages before the CTA exits
        const uint32_t first = i > static_cast<uint32_t>(kStages) ? i - kStages : 0u;
        for (uint32_t j = first; j < i; ++j)
          mbar_wait(base + S::full + 8 * (j % kStages), (j / kStages) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      uint32_t i = 0;
      bool ok = true;
      for (int k = 0; k < count && ok; ++k) {
        const int g = k & 1;
        for (int grp = 0; grp < ngroups && ok; ++grp) {
          const uint32_t use = static_cast<uint32_t>((k >> 1) * ngroups + grp);
          if (!wait_here(base + S::tempty + 8 * g, (use & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int pl = 0; pl < GS && grp * GS + pl < P && ok; ++pl)
            for (int c = 0; c < NC; ++c, ++i) {
              const uint32_t s = i % kStages, ph = (i / kStages) & 1u;
              if (!wait_here(base + S::full + 8 * s, ph, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t d = tmem + g * kHalfCols + pl * NB + c * 64;
              const uint32_t atile = base + S::stages + s * kAtomBytes;
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                mma_f8f6f4(d, sw64_desc(atile + 32 * kk), sw64_desc(base + S::hmat + 32 * kk),
                           kIdesc, kk > 0 ? 1u : 0u);
              mma_commit(base + S::empty + 8 * s);   // the stage is free once these are done
            }
          if (ok) mma_commit(base + S::tfull + 8 * g);
        }
      }
      // every MMA of this CTA has completed before the tensor memory is freed
      mma_commit(base + S::mma_done);
      mbar_wait(base + S::mma_done, 0);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue ----
    const int g = (warp - 2) >> 2;               // group: half g, tiles k % 2 == g
    const int quad = warp & 3;                   // TMEM lanes 32 quad .. 32 quad + 31
    const int row = quad * 32 + lane;            // block row of the tile
    const bool leader = (warp == 2 + 4 * g) && lane == 0;
    const uint32_t thalf = tmem + (static_cast<uint32_t>(quad * 32) << 16) + g * kHalfCols;
    const uint32_t staging = base + S::out + g * NC * kOutAtomBytes;
    if (leader) prefetch_map(&maps.out);
    bool stop = false;

    // (alpha, s) pairs of one shard group of one tile, read one group ahead of
    // their use so that the global-memory latency overlaps a group's work
    float2 nxt[GS];
    auto fetch = [&](int kk, int gg) {
      const int64_t bb = (blockIdx.x + static_cast<int64_t>(kk) * G) * kRows + row;
#pragma unroll
      for (int pl = 0; pl < GS; ++pl) {
        const int p = gg * GS + pl;
        nxt[pl] = make_float2(1.0f, 0.0f);   // d = 0 for absent shards and rows
        if (kk < count && p < P && bb < nblocks)
          nxt[pl] = __ldg(reinterpret_cast<const float2*>(a.shard[p] + a.scales_off) + bb);
      }
    };
    fetch(g, 0);

    for (int k = g; k < count && !stop; k += 2) {
      const int64_t tile = blockIdx.x + static_cast<int64_t>(k) * G;

      float z[NC][64];
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int i = 0; i < 64; ++i) z[c][i] = 0.0f;

      for (int grp = 0; grp < ngroups; ++grp) {
        // scales of this group's shards: d = s / alpha / sqrt(n)
        float2 cur[GS];
#pragma unroll
        for (int pl = 0; pl < GS; ++pl) cur[pl] = nxt[pl];
        if (grp + 1 < ngroups) {
          fetch(k, grp + 1);
        } else {
          fetch(k + 2, 0);
        }
        float d[GS];
#pragma unroll
        for (int pl = 0; pl < GS; ++pl) d[pl] = __fdividef(cur[pl].y, cur[pl].x) * a.inv_sqrt_n;
        const uint32_t use = static_cast<uint32_t>((k >> 1) * ngroups + grp);
        const bool got = wait_here(base + S::tfull + 8 * g, use & 1u, abort_flag);
        if (leader && grp == 0) bulk_wait_read<0>();   // the group's last store has read the staging
        if (group_any(1 + g, !got || *abort_flag != 0u)) {
          stop = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int pl = 0; pl < GS; ++pl) {
          if (grp * GS + pl >= P) break;
          const f2 d2{d[pl], d[pl]};
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int h = 0; h < 64 / kLoadCols; ++h) {
              float v[kLoadCols];
#pragma unroll
              for (int q = 0; q < kLoadCols / 16; ++q)
                tmem_ld16(thalf + pl * NB + c * 64 + h * kLoadCols + q * 16, v + q * 16);
              tmem_wait_ld();
#pragma unroll
              for (int q = 0; q < kLoadCols / 16; ++q) reg_fence16(v + q * 16);
#pragma unroll
              for (int i = 0; i < kLoadCols; i += 2) {
                const int e = h * kLoadCols + i;
                const f2 r = fma2(d2, f2{v[i], v[i + 1]}, f2{z[c][e], z[c][e + 1]});
                z[c][e] = r.x;
                z[c][e + 1] = r.y;
              }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(base + S::tempty + 8 * g);
      }
      if (stop) break;

      // remaining rotation levels across the chunks: x_hat = (H_NC (x) I) z
#pragma unroll
      for (int m = 1; m < NC; m <<= 1)
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if ((c & m) == 0) {
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
              const f2 x0{z[c][i], z[c][i + 1]}, x1{z[c + m][i], z[c + m][i + 1]};
              const f2 s = add2(x0, x1), t = sub2(x0, x1);
              z[c][i] = s.x;
              z[c][i + 1] = s.y;
              z[c + m][i] = t.x;
              z[c + m][i + 1] = t.y;
            }
          }

      // bf16 into the staging atoms: row `row` of atom c is 128 bytes, its
      // 16-byte pieces permuted by the 128-byte swizzle (piece ^= row & 7)
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int piece = 0; piece < 8; ++piece) {
          const int i = piece * 8;
          const uint4 w = make_uint4(pack_bf16x2(z[c][i], z[c][i + 1]), pack_bf16x2(z[c][i + 2], z[c][i + 3]),
                                     pack_bf16x2(z[c][i + 4], z[c][i + 5]), pack_bf16x2(z[c][i + 6], z[c][i + 7]));
          sts128(staging + c * kOutAtomBytes + row * 128 + 16 * (piece ^ (row & 7)), w);
        }
      fence_proxy_async_smem();   // the tile is visible to the tensor store
      group_sync(1 + g);
      if (leader) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
          tma_store_2d(&maps.out, staging + c * kOutAtomBytes, c * 64, static_cast<int>(tile * kRows));
        bulk_commit();
      }
    }
    if (leader) bulk_wait_read<0>();   // every store has read the staging (the kernel's end
                                       // makes the stored output visible)
  }

  // ---- tear-down: free the tensor memory ----
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t decompress_mma_smem_bytes(int block) {
  return block == 64 ? DSmem<64>::bytes : DSmem<128>::bytes;
}

const void* decompress_mma_kernel_ptr(int block) {
  return block == 64 ? reinterpret_cast<const void*>(decompress_mma_kernel<64>)
                     : reinterpret_cast<const void*>(decompress_mma_kernel<128>);
}

cudaError_t launch_decompress_mma(const DecompressArgs& a, int block, int grid, cudaStream_t stream) {
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  DmmaMaps maps;
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kRows)};
  const cuuint32_t unit[2] = {1, 1};
  const cuuint64_t dim[2] = {static_cast<cuuint64_t>(block), static_cast<cuuint64_t>(a.nblocks)};
  const cuuint64_t cstride[1] = {static_cast<cuuint64_t>(block)};
  for (int p = 0; p < a.P; ++p) {
    if (encode(&maps.codes[p], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.shard[p]), dim,
               cstride, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  for (int p = a.P; p < TACO_MAX_SHARDS; ++p) maps.codes[p] = maps.codes[0];
  const cuuint64_t ostride[1] = {static_cast<cuuint64_t>(block) * 2};
  if (encode(&maps.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out, dim, ostride, box, unit,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = decompress_mma_smem_bytes(block);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void (*kern)(DmmaMaps, DecompressArgs) = block == 64 ? decompress_mma_kernel<64> : decompress_mma_kernel<128>;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t decompress_mma_fault(unsigned int* bits, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_decompress_mma_fault, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_decompress_mma_fault, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace taco

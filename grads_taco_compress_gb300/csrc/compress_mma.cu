// TACO fused compress on the 5th-generation tensor cores (tcgen05 + TMEM):
// taco_compress_shards_mma and the INT8 fallback's compress. Same outputs as
// the CUDA-core FWHT of compress.cu, within the parity bar, and faster on
// every measured shape.
//
// The operator is the one of compress.cu ("TACO: Efficient Communication
// Compression of Intermediate Tensors ...", gist.science pt summary, §2.B.1
// ASH, §2.B.2 DS, §2.B.3 one fused kernel). What changes is where the
// Hadamard products run. Sylvester's construction gives
//   H_n = H_{n/64} (x) H_64,   element e = 64 * chunk + i,
// so a block of n = 64 * NC elements is rotated in two steps:
//   1. every 64-element chunk u_c = H_64 x_c is one row of a dense product
//      D[128 x 64] = A[128 x 64] * H_64^T on the tensor cores: A holds one
//      chunk of 128 consecutive blocks (bf16, exact), H_64 is +-1 (exact in
//      bf16), D accumulates in fp32 in tensor memory;
//   2. t = (H_NC (x) I_64) u, NC - 1 butterfly levels across the chunks,
//      done in registers by the thread that owns the block.
// The energy comes from the rotated block (Parseval: sum t^2 = n sum x^2),
// so no thread reads x itself: alpha = n sqrt(E*) / sqrt(sum t^2).
//
// CTA = 11 warps, one per SM (its registers do not fit twice), with a ring of
// 5 input stages for n = 64 and 6 for n = 128 and 256, the fastest shapes
// measured with the tile schedule below (4, 7 and 8 stages were slower):
//   warp 0     TMA producer: 3-D tensor loads of [128 blocks x 64 elements]
//              bf16 atoms (16 KB, 128-byte swizzle) into a ring of stages;
//   warp 1     owns the tensor memory (2 accumulators x n columns) and one
//              lane issues the MMAs (4 x K=16 per atom), committing each atom
//              to its stage's "empty" barrier and each tile to "full";
//   warps 2-9  two epilogue groups of 4 warps; group g takes the CTA's tiles
//              k with k % 2 == g from accumulator g. Thread (warp w, lane l)
//              owns block row 32 (w % 4) + l of the tile (the TMEM lanes a
//              warp may read). It loads its row with tcgen05.ld, finishes the
//              rotation, computes alpha, s and the codes, writes the codes
//              into a 64-byte-swizzled staging buffer that one thread stores
//              with 3-D TMA tensor stores, and stores its (alpha, s) pair;
//              each warp then folds its rows' largest s and count of s > 1
//              into the CTA's totals for the tile's shard (shared memory);
//   warp 10    tile scheduler (below); once the pool is dry it also makes the
//              CTA's per-tensor header arrivals, overlapping the last tiles.
// Tile schedule: the CTAs of shard y (gridDim.x of them, blockIdx.y == y)
// take 3/4 of the per-CTA share of that shard's tiles round-robin (tile
// blockIdx.x + k * gridDim.x), then every CTA claims the rest of all shards'
// tiles one at a time from one counter in the workspace (shard 0's tile
// word), shards interleaved. So the CTAs that stream faster take more, and
// the CTAs of a launch finish together: with a static split the spread of
// per-SM progress grew through the launch to several tiles, and with one
// pool per shard whole shards finished apart (gpt3-6.7b-grad: the median
// CTA of the slowest shard 6 us after that of the fastest). The scheduler
// lane keeps two claims ready in a shared-memory ring, which hides the
// atomic's round trip from the producer. A tile travels as one int, its
// shard in bits 24 and up (a tile index needs 24 bits); it reaches the MMA
// lane with the barrier of its first atom and the epilogue group with the
// group's `info` barrier; a -1 ends every role.
// Before it waits for the preceding grid, the producer asks L2 for the
// tiles of its first ring of stages (a prefetch returns no data, so it is
// safe before that grid's writes are visible): the launch's first loads
// then find their data in L2 instead of waiting a DRAM round trip.
// FMT selects the code format: 0 = FP8 E4M3 (Q_max 448), 1 = the INT8
// fallback (Q_max 127, round half to even; pt summary §5, hardware without
// FP8).
// Every wait is bounded in time; a wait that gives up sets a CTA-wide abort
// flag that ends every role's loop, records kFaultCompressMmaWait and lets
// the CTA drain its copies and MMAs before it frees the tensor memory.

#include <cmath>
#include <mutex>

#include "taco_launch.h"
#include "tcgen05.cuh"

namespace taco {

namespace {

__device__ unsigned int g_compress_mma_fault;

// The per-tensor header of this kernel. Workspace of a shard (16 bytes,
// zero between calls):
//   [u64: arrivals << 48 | count of s > 1][u32 running max-s bits][u32 tile claims]
// A CTA's largest s is folded into the running maximum (an atomic max on
// the float's bits, which order like the values because every s is positive
// and fmaxf drops NaN), and a release fence follows it. The count of s > 1
// rides on the CTA's arrival: one 64-bit add that counts the CTA and adds
// the count, so the count needs no ordering of its own, and the fence before
// it makes that add a release for the maximum; the add is an acquire. The
// arrival that completes the count takes the maximum with one exchange that
// zeroes it, writes the header and resets the counter and the tile word.
constexpr int kArrivalShift = 48;   // arrivals above, the count of s > 1 below

__device__ __forceinline__ void fold_max(float m, uint8_t* ws_shard) {
  if (m > 0.0f)
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(ws_shard + 8), "r"(__float_as_uint(m))
                 : "memory");
}
__device__ __forceinline__ void release_fence() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// after a release fence of this thread that follows every fold of the CTA
__device__ __forceinline__ void arrive(uint32_t n, uint32_t arrivals, uint8_t* ws_shard, taco_header* hd,
                                       int64_t N, int64_t h, int block, int variant, float target_energy,
                                       float q_max) {
  unsigned long long old;
  asm volatile("atom.add.acquire.gpu.global.u64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(ws_shard), "l"((1ull << kArrivalShift) + n)
               : "memory");
  if ((old >> kArrivalShift) != arrivals - 1u) return;
  uint32_t m;
  asm volatile("atom.exch.relaxed.gpu.global.b32 %0, [%1], 0;" : "=r"(m) : "l"(ws_shard + 8) : "memory");
  write_header(hd, N, h, block, variant, target_energy, q_max, __uint_as_float(m),
               static_cast<uint32_t>((old & ((1ull << kArrivalShift) - 1)) + n));
  // leaves the workspace zero-filled for the next call: the counter and the
  // tile word (every claim of the launch came before the arrivals)
  *reinterpret_cast<volatile unsigned long long*>(ws_shard) = 0ull;
  *reinterpret_cast<volatile uint32_t*>(ws_shard + 12) = 0u;
}

constexpr int kRows = 128;                    // blocks per tile (the MMA's M)
constexpr int kRing = 8;                      // tile indices in flight, producer -> MMA lane
constexpr int kClaims = 2;                    // claimed tiles in flight, scheduler -> producer
constexpr uint32_t kAtomBytes = kRows * 64 * 2;       // 16 KB of bf16
constexpr uint32_t kCodeAtomBytes = kRows * 64;       // 8 KB of codes
constexpr uint32_t kHBytes = 64 * 64 * 2;             // H_64 in bf16
constexpr int kItemShift = 24;                        // tile item: shard << 24 | tile
static_assert((kMmaMaxBlocks + kRows - 1) / kRows < (int64_t{1} << kItemShift) &&
                  (int64_t{TACO_MAX_SHARDS} << kItemShift) <= INT32_MAX,
              "a tile item fits an int");

// Shared memory map (offsets from a 1024-byte aligned base) and CTA shape.
template <int NB>
struct Smem {
  static constexpr int NC = NB / 64;
  static constexpr int NG = compress_mma_groups(NB);               // epilogue groups
  static constexpr int threads = compress_mma_threads(NB);
  static constexpr int kStages = NB == 64 ? 5 : 6;                  // 16 KB atoms in flight
  static constexpr uint32_t stages = 0;
  static constexpr uint32_t hmat = stages + kStages * kAtomBytes;
  static constexpr uint32_t codes = hmat + kHBytes;                 // [group][chunk] atoms
  static constexpr uint32_t bars = codes + NG * NC * kCodeAtomBytes;
  // barriers: full[kStages], empty[kStages], tfull[NG], tempty[NG], info[NG],
  // cfull[kClaims], cempty[kClaims], mma_done, hdr_ready
  static constexpr uint32_t full = bars;
  static constexpr uint32_t empty = full + 8 * kStages;
  static constexpr uint32_t tfull = empty + 8 * kStages;
  static constexpr uint32_t tempty = tfull + 8 * NG;
  static constexpr uint32_t info = tempty + 8 * NG;
  static constexpr uint32_t cfull = info + 8 * NG;
  static constexpr uint32_t cempty = cfull + 8 * kClaims;
  static constexpr uint32_t mma_done = cempty + 8 * kClaims;
  static constexpr uint32_t hdr_ready = mma_done + 8;              // every epilogue warp's share is in
  static constexpr uint32_t tmem_slot = hdr_ready + 8;
  static constexpr uint32_t abort_flag = tmem_slot + 4;
  static constexpr uint32_t tile_ring = abort_flag + 4;   // int[kRing]: tile of the CTA's tile k
  static constexpr uint32_t tile_of = tile_ring + 4 * kRing;      // int[NG]: tile of accumulator g
  static constexpr uint32_t claim = tile_of + 4 * NG;             // int[kClaims]: claimed tiles
  static constexpr uint32_t n_tiles = claim + 4 * kClaims;         // int: the CTA's tiles, -1 until known
  // u32[TACO_MAX_SHARDS] each: the CTA's largest s bits and count of s > 1 per shard
  static constexpr uint32_t hdr_max = n_tiles + 4;
  static constexpr uint32_t hdr_cnt = hdr_max + 4 * TACO_MAX_SHARDS;
  static constexpr uint32_t end = hdr_cnt + 4 * TACO_MAX_SHARDS;
  static constexpr uint32_t bytes = end + 1024;                     // + alignment slack
};

// Instruction descriptor: bf16 A and B, fp32 D, M = 128, N = 64.
constexpr uint32_t kIdesc = instr_desc(1, kRows, 64);

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return umma_desc(saddr, kSwizzle128, 1024);
}

__device__ __forceinline__ bool wait_here(uint32_t bar, uint32_t parity,
                                          volatile uint32_t* abort_flag) {
  return wait_or_abort(bar, parity, abort_flag, &g_compress_mma_fault, kFaultCompressMmaWait);
}

// ------------------------------------------------------------- epilogue ----
// Values of one slice of the thread's block: u[c][i] = column (slice * SL + i)
// of chunk c. After the butterflies, u[c][i] is element 64 c + slice * SL + i
// of t = H_n x.
template <int NC, int SL>
__device__ __forceinline__ void load_slice(uint32_t tacc, int slice, float (&u)[NC][SL]) {
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int q = 0; q < SL / 16; ++q)
      tmem_ld16(tacc + c * 64 + slice * SL + q * 16, &u[c][q * 16]);
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int q = 0; q < SL / 16; ++q) reg_fence16(&u[c][q * 16]);
}

// t = (H_NC (x) I) u over the chunk index, in place.
template <int NC, int SL>
__device__ __forceinline__ void chunk_butterflies(float (&u)[NC][SL]) {
#pragma unroll
  for (int m = 1; m < NC; m <<= 1)
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if ((c & m) == 0) {
#pragma unroll
        for (int i = 0; i < SL; i += 2) {
          const f2 a{u[c][i], u[c][i + 1]}, b{u[c + m][i], u[c + m][i + 1]};
          const f2 s = add2(a, b), d = sub2(a, b);
          u[c][i] = s.x;
          u[c][i + 1] = s.y;
          u[c + m][i] = d.x;
          u[c + m][i + 1] = d.y;
        }
      }
}

// Running sum of squares (four packed accumulators) and max / min.
template <int NC, int SL>
__device__ __forceinline__ void slice_stats(const float (&u)[NC][SL], f2 (&ea)[4], float (&hi)[4],
                                            float (&lo)[4]) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
#pragma unroll
    for (int i = 0; i < SL; i += 2) {
      const f2 v{u[c][i], u[c][i + 1]};
      ea[(i >> 1) & 3] = fma2(v, v, ea[(i >> 1) & 3]);
    }
#pragma unroll
    for (int i = 0; i < SL; i += 4) {
      const int j = (i >> 2) & 3;
      hi[j] = max3(hi[j], max3(u[c][i], u[c][i + 1], u[c][i + 2]), u[c][i + 3]);
      lo[j] = min3(lo[j], min3(u[c][i], u[c][i + 1], u[c][i + 2]), u[c][i + 3]);
    }
  }
}

// u *= 2^-k (two exact power-of-two factors).
template <int NC, int SL>
__device__ __forceinline__ void scale_slice(float (&u)[NC][SL], f2 s1, f2 s2) {
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < SL; i += 2) {
      const f2 t = mul2(mul2(f2{u[c][i], u[c][i + 1]}, s1), s2);
      u[c][i] = t.x;
      u[c][i + 1] = t.y;
    }
}

// Codes of one slice into the group's staging atoms: chunk c of block row
// `row` is 64 bytes at row * 64 of atom c, its 16-byte pieces permuted by the
// 64-byte swizzle (piece ^= (row >> 1) & 3) that the tensor store undoes.
template <int NC, int SL, int FMT, bool CLAMP>
__device__ __forceinline__ void slice_codes(const float (&u)[NC][SL], int slice, float g,
                                            uint32_t stage_codes, int row) {
  const f2 g2{g, g};
  const uint32_t rbase = stage_codes + row * 64;
  const int sw = (row >> 1) & 3;
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int q = 0; q < SL / 16; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = q * 16 + 4 * k;
        const f2 y0 = mul2(f2{u[c][i], u[c][i + 1]}, g2);
        const f2 y1 = mul2(f2{u[c][i + 2], u[c][i + 3]}, g2);
        w[k] = (FMT == 0) ? e4m3x4_from_f32(y0.x, y0.y, y1.x, y1.y) : i8x4_from_f32<CLAMP>(y0, y1);
      }
      const int piece = (slice * SL) / 16 + q;
      sts128(rbase + c * kCodeAtomBytes + 16 * (piece ^ sw), make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// How far the tensor cores' fp32 image t = H_n x of a block is used, by its
// largest magnitude max |t| (>= max |x|, and 0 only for an all-zero block).
// The tensor cores keep bf16 subnormal inputs and fp32 subnormal sums exact
// (measured), and no partial sum of a block overflows while max |t| <= 2^119
// (each is at most n max |x| <= 2^127).
//   [2^-40, 2^56] or 0: t is squared and summed as it is (the squares that
//       fall into fp32's subnormal range weigh less than 2^-60 of the sum);
//   [2^-120, 2^119] otherwise: the sum of squares is taken again from
//       tensor memory with t scaled by 2^-k (k = the exponent of max |t|,
//       exact) and 2^-k goes back into alpha; t itself is used as it is
//       (its subnormal grid is below 2^-29 max |t|, finer than a code);
//   anything else (a block of bf16 subnormals only, or one whose rotation
//       overflowed fp32): done again from x in global memory (exact_block).
constexpr float kTrustLo = 0x1p-40f;
constexpr float kTrustHi = 0x1p56f;
constexpr float kRescaleLo = 0x1p-120f;
constexpr float kRescaleHi = 0x1p119f;

// One block from its bf16 values in global memory, for the thread that owns
// its row of the tile: x scaled by 2^-k (k the exponent of max |x|, exact),
// the energy from the scaled values, alpha = 2^-k sqrt(n E*) / sqrt(sum x'^2)
// kept in [2^-126, 2^126], and the Hadamard transform t' of the scaled block
// in fp32; the rotated values are then alpha 2^k t' / sqrt(n) for any
// magnitude of x. Writes the block's codes into the row of the staging atoms
// (the layout slice_codes writes) and returns (alpha, s). Rare by
// construction, so it keeps the block in local memory and leaves the
// register budget of the fast path alone.
template <int NB, int VARIANT, int FMT>
__device__ __noinline__ float2 exact_block(const uint16_t* __restrict__ xb, float sqrt_nE,
                                           float inv_sqrt_n, float s_static, uint32_t stage_codes,
                                           int row) {
  constexpr float QMAX = (FMT == 0) ? 448.0f : 127.0f;
  float v[NB];
  float m = 0.0f;
#pragma unroll 1
  for (int i = 0; i < NB; i += 64) {
    uint4 w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) w[q] = __ldg(reinterpret_cast<const uint4*>(xb + i) + q);   // 8 loads in flight
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        v[i + 8 * q + 2 * r] = bf16_lo(ws[r]);
        v[i + 8 * q + 2 * r + 1] = bf16_hi(ws[r]);
        m = max3(m, fabsf(bf16_lo(ws[r])), fabsf(bf16_hi(ws[r])));
      }
    }
  }
  float alpha = 1.0f, c = 0.0f, tm = 0.0f;
  if (m > 0.0f) {
    const int k = ilogbf(m);                  // m 2^-k in [1, 2)
    f2 ea[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 1
    for (int i = 0; i < NB; i += 8) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const f2 xs{ldexpf(v[i + 2 * q], -k), ldexpf(v[i + 2 * q + 1], -k)};
        v[i + 2 * q] = xs.x;
        v[i + 2 * q + 1] = xs.y;
        ea[q] = fma2(xs, xs, ea[q]);
      }
    }
    const f2 e01 = add2(ea[0], ea[1]), e23 = add2(ea[2], ea[3]);
    alpha = alpha_scaled(sqrt_nE, (e01.x + e01.y) + (e23.x + e23.y), k);
    c = ldexpf(alpha, k) * inv_sqrt_n;        // rotated value = c t'
#pragma unroll 1
    for (int hs = 1; hs < NB; hs <<= 1)       // Sylvester order: t_j = sum_i (-1)^popc(i&j) x_i
#pragma unroll 1
      for (int i = 0; i < NB; i += 2 * hs)
#pragma unroll 1
        for (int j = i; j < i + hs; ++j) {
          const float p = v[j], q = v[j + hs];
          v[j] = p + q;
          v[j + hs] = p - q;
        }
#pragma unroll 1
    for (int i = 0; i < NB; ++i) tm = fmaxf(tm, fabsf(v[i]));
  }
  const float amax = c * tm;
  const float sc = (VARIANT == 0)   ? fmaxf(1.0f, amax * (1.0f / QMAX))
                   : (VARIANT == 1) ? (amax > 0.f ? amax * (1.0f / QMAX) : 1.0f)
                                    : s_static;
  const float g = __fdividef(c, sc);
  const f2 g2{g, g};
  const uint32_t rbase = stage_codes + row * 64;
  const int sw = (row >> 1) & 3;
#pragma unroll 1
  for (int i = 0; i < NB; i += 16) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const f2 y0 = mul2(f2{v[i + 4 * q], v[i + 4 * q + 1]}, g2);
      const f2 y1 = mul2(f2{v[i + 4 * q + 2], v[i + 4 * q + 3]}, g2);
      w[q] = (FMT == 0) ? e4m3x4_from_f32(y0.x, y0.y, y1.x, y1.y) : i8x4_from_f32<VARIANT == 2>(y0, y1);
    }
    const int chunk = i >> 6, piece = (i & 63) >> 4;
    sts128(rbase + chunk * kCodeAtomBytes + 16 * (piece ^ sw), make_uint4(w[0], w[1], w[2], w[3]));
  }
  return make_float2(alpha, sc);
}

template <int NB, int VARIANT, int FMT>
__global__ void __launch_bounds__(Smem<NB>::threads, 1)
compress_mma_kernel(const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_codes, CompressArgs a) {
  using S = Smem<NB>;
  constexpr int NC = NB / 64;            // 64-element chunks per block
  constexpr int SL = 64 / NC;            // columns per slice (64 registers per slice)
  constexpr int NG = S::NG;
  constexpr int kThreads = S::threads;
  constexpr int kStages = S::kStages;
  constexpr int kSchedWarp = 2 + 4 * NG;
  // the producer writes tile k's ring slot after the empty waits of tile k-1,
  // so the MMA lane has read every slot up to k - kRing by then
  static_assert(kRing * NC >= kStages + 1, "a tile index is read before its ring slot is rewritten");
  constexpr uint32_t TMEM_COLS = NG * NB;   // one accumulator per epilogue group
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "tensor memory columns");
  constexpr float QMAX = (FMT == 0) ? 448.0f : 127.0f;

  extern __shared__ unsigned char smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* const sbase = smem_raw + (base - smem_u32(smem_raw));
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sbase + S::abort_flag);
  volatile int* tile_ring = reinterpret_cast<volatile int*>(sbase + S::tile_ring);
  volatile int* tile_of = reinterpret_cast<volatile int*>(sbase + S::tile_of);
  volatile int* claim = reinterpret_cast<volatile int*>(sbase + S::claim);
  volatile int* n_tiles = reinterpret_cast<volatile int*>(sbase + S::n_tiles);
  unsigned int* const hdr_max = reinterpret_cast<unsigned int*>(sbase + S::hdr_max);
  unsigned int* const hdr_cnt = reinterpret_cast<unsigned int*>(sbase + S::hdr_cnt);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int shard = blockIdx.y;
  const int P = gridDim.y;
  const int64_t nblocks = a.nblocks;
  const int64_t ntiles = (nblocks + kRows - 1) / kRows;
  const int64_t G = gridDim.x;
  // round-robin tiles per CTA: 3/4 of the even share, rounded up (a CTA with
  // one tile starts it without waiting for a claim); n_static * G <= ntiles
  const int n_static = static_cast<int>((3 * (ntiles / G) + 3) / 4);

  // ---- set-up: barriers, H_64, tensor memory ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(base + S::full + 8 * s, 1);
      mbar_init(base + S::empty + 8 * s, 1);
    }
    for (int g = 0; g < NG; ++g) {
      mbar_init(base + S::tfull + 8 * g, 1);
      mbar_init(base + S::tempty + 8 * g, 4);   // one arrival per epilogue warp
      mbar_init(base + S::info + 8 * g, 1);
    }
    for (int c = 0; c < kClaims; ++c) {
      mbar_init(base + S::cfull + 8 * c, 1);
      mbar_init(base + S::cempty + 8 * c, 1);
    }
    mbar_init(base + S::mma_done, 1);
    mbar_init(base + S::hdr_ready, 4 * NG);   // one arrival per epilogue warp
    *n_tiles = -1;
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (threadIdx.x < 2 * TACO_MAX_SHARDS) hdr_max[threadIdx.x] = 0u;   // hdr_cnt follows hdr_max
  // H_64 (entries (-1)^popcount(r & k)) as B: 64 rows of 128 bytes, K-major,
  // 16-byte pieces swizzled by (row & 7).
  for (int p = threadIdx.x; p < 64 * 8; p += kThreads) {
    const int r = p >> 3, piece = p & 7;
    uint32_t w[4];
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
      const int k0 = piece * 8 + 2 * k2;
      const uint32_t lo = (__popc(r & k0) & 1) ? 0xBF80u : 0x3F80u;
      const uint32_t hi = (__popc(r & (k0 + 1)) & 1) ? 0xBF80u : 0x3F80u;
      w[k2] = lo | (hi << 16);
    }
    sts128(base + S::hmat + r * 128 + 16 * (piece ^ (r & 7)), make_uint4(w[0], w[1], w[2], w[3]));
  }
  fence_proxy_async_smem();   // H is read by the tensor cores (async proxy)
  if (warp == 1) tmem_alloc(base + S::tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = lds_u32(base + S::tmem_slot);

  grid_launch_dependents();
  if (warp == 0 && lane == 0) {
    prefetch_map(&map_x);
    // the tiles of the first ring of stages into L2 while the preceding grid
    // finishes (no data reaches this CTA before the wait below)
    const int npf = min(n_static, (kStages + NC - 1) / NC);
    for (int k = 0; k < npf; ++k)
      for (int c = 0; c < NC; ++c)
        tma_prefetch_3d(&map_x, c * 64, static_cast<int>((blockIdx.x + k * G) * kRows), shard);
  }
  grid_dependency_wait();   // no global access before the preceding grid is done

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer ----
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      uint32_t i = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int tile;   // the tile item: shard << kItemShift | tile, or -1
        if (k < n_static) {
          tile = (shard << kItemShift) | static_cast<int>(blockIdx.x + static_cast<int64_t>(k) * G);
        } else {
          const uint32_t j = static_cast<uint32_t>(k - n_static), c = j % kClaims;
          if (!wait_here(base + S::cfull + 8 * c, (j / kClaims) & 1u, abort_flag)) break;
          tile = claim[c];
          mbar_arrive(base + S::cempty + 8 * c);
          if (tile < 0) *n_tiles = k;   // the CTA's tile count, for the epilogue's last tiles
        }
        tile_ring[k % kRing] = tile;   // published by the arrival on the first atom's barrier
        for (int c = 0; c < (tile < 0 ? 1 : NC); ++c, ++i) {
          const uint32_t s = i % kStages, ph = (i / kStages) & 1u;
          if (!wait_here(base + S::empty + 8 * s, ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (tile < 0) {
            mbar_arrive(base + S::full + 8 * s);   // the end: an arrival without a copy
          } else {
            mbar_arrive_expect_tx(base + S::full + 8 * s, kAtomBytes);
            tma_load_3d(base + S::stages + s * kAtomBytes, &map_x, c * 64,
                        (tile & ((1 << kItemShift) - 1)) * kRows, tile >> kItemShift,
                        base + S::full + 8 * s, policy);
          }
        }
        if (tile < 0) break;
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
      for (int k = 0; ok; ++k) {
        const int g = k % NG;
        const uint32_t use = static_cast<uint32_t>(k / NG);
        if (!wait_here(base + S::tempty + 8 * g, (use & 1u) ^ 1u, abort_flag)) break;
        tc_fence_after();
        if (!wait_here(base + S::full + 8 * (i % kStages), (i / kStages) & 1u, abort_flag)) break;
        // the tile of local tile k goes on to its epilogue group, whose
        // accumulator (and tile_of slot) is free
        const int tile = tile_ring[k % kRing];
        tile_of[g] = tile;
        mbar_arrive(base + S::info + 8 * g);
        if (tile < 0) {
          // the end: the other groups learn it once their accumulators are free
          for (int j = 1; j < NG; ++j) {
            const int g2 = (k + j) % NG;
            const uint32_t use2 = static_cast<uint32_t>((k + j) / NG);
            if (!wait_here(base + S::tempty + 8 * g2, (use2 & 1u) ^ 1u, abort_flag)) break;
            tile_of[g2] = -1;
            mbar_arrive(base + S::info + 8 * g2);
          }
          break;
        }
        for (int c = 0; c < NC; ++c, ++i) {
          const uint32_t s = i % kStages, ph = (i / kStages) & 1u;
          if (c > 0 && !wait_here(base + S::full + 8 * s, ph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + g * NB + c * 64;
          const uint32_t atile = base + S::stages + s * kAtomBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(d, sw128_desc(atile + 32 * kk), sw128_desc(base + S::hmat + 32 * kk), kIdesc,
                    kk > 0 ? 1u : 0u);
          mma_commit(base + S::empty + 8 * s);   // the stage is free once these MMAs are done
        }
        if (ok) mma_commit(base + S::tfull + 8 * g);
      }
      // every MMA of this CTA has completed before the tensor memory is freed
      mma_commit(base + S::mma_done);
      mbar_wait(base + S::mma_done, 0);
    }
    __syncwarp();
  } else if (warp == kSchedWarp) {
    // ---------------------------------------------------- tile scheduler ----
    if (lane == 0) {
      // one pool for the whole launch: shard 0's tile word; item j of the
      // pool is tile first + j / P of shard j % P
      unsigned int* next = reinterpret_cast<unsigned int*>(a.workspace) + 3;
      const int64_t first = static_cast<int64_t>(n_static) * G;   // first tile of each shard's pool
      const int64_t pool = (ntiles - first) * P;
      for (uint32_t j = 0;; ++j) {
        const uint32_t c = j % kClaims;
        if (!wait_here(base + S::cempty + 8 * c, ((j / kClaims) & 1u) ^ 1u, abort_flag)) break;
        const int64_t t = atomicAdd(next, 1u);
        const int tile = t < pool ? (static_cast<int>(t % P) << kItemShift) | static_cast<int>(first + t / P)
                                  : -1;
        claim[c] = tile;
        mbar_arrive(base + S::cfull + 8 * c);
        if (tile < 0) break;
      }
    }
    __syncwarp();
    // The per-tensor headers; lane p handles shard p. Every CTA arrives on
    // every shard (a CTA may have compressed tiles of any shard), and the
    // last of the G * P arrivals writes the header. With the pool dry, the
    // largest s the CTA has seen so far goes into the shard's running
    // maximum and a release fence follows, while the last tiles are still on
    // their way. Once every epilogue warp has folded in its last tile
    // (hdr_ready), the arrival carries the count of s > 1; a second fold and
    // fence come before it only if the CTA's largest s grew meanwhile. After
    // a wait that gave up the arrivals still happen, so that the workspace
    // is reset.
    uint8_t* const ws_p = a.workspace + lane * kWorkspaceShardStride;
    float m_early = 0.0f;
    if (lane < P) {
      m_early = __uint_as_float(reinterpret_cast<volatile unsigned int*>(hdr_max)[lane]);
      fold_max(m_early, ws_p);
      release_fence();
    }
    wait_here(base + S::hdr_ready, 0, abort_flag);
    if (lane < P) {
      const float m = __uint_as_float(hdr_max[lane]);
      if (m > m_early) {
        fold_max(m, ws_p);
        release_fence();
      }
      arrive(hdr_cnt[lane], G * P, ws_p, a.headers + lane, a.N, a.h, NB, VARIANT, a.target_energy, QMAX);
    }
  } else {
    // -------------------------------------------------------- epilogue ----
    const int g = (warp - 2) >> 2;               // group: accumulator and tiles k % NG == g
    const int quad = warp & 3;                   // TMEM lanes 32 quad .. 32 quad + 31
    const int row = quad * 32 + lane;            // block row of the tile
    const bool leader = (warp == 2 + 4 * g) && lane == 0;
    const uint32_t tacc = tmem + (static_cast<uint32_t>(quad * 32) << 16) + g * NB;
    const uint32_t staging = base + S::codes + g * NC * kCodeAtomBytes;
    if (leader) prefetch_map(&map_codes);
    // the warp's share of its tile's shard header: the largest s (bits of a
    // positive float order like its value; fmaxf drops NaN) and the count
    // of s > 1, into the CTA's per-shard totals
    auto fold_header = [&](int ts, bool valid, float sc) {
      const uint32_t wmax = __reduce_max_sync(kFullMask, valid ? __float_as_uint(fmaxf(sc, 0.0f)) : 0u);
      const uint32_t wcnt = __popc(__ballot_sync(kFullMask, valid && sc > 1.0f));
      if (lane == 0) {
        atomicMax(hdr_max + ts, wmax);
        atomicAdd(hdr_cnt + ts, wcnt);
      }
    };
    bool shared_all = false;   // the warp has arrived on hdr_ready

    for (int k = g;; k += NG) {
      const uint32_t use = static_cast<uint32_t>(k / NG);
      const bool got_info = wait_here(base + S::info + 8 * g, use & 1u, abort_flag);
      const int tile_k = tile_of[g];
      if (group_any(1 + g, !got_info || tile_k < 0 || *abort_flag != 0u)) break;
      const bool got = wait_here(base + S::tfull + 8 * g, use & 1u, abort_flag);
      if (leader) bulk_wait_read<0>();           // the group's last store has read the staging
      if (group_any(1 + g, !got || *abort_flag != 0u)) break;
      tc_fence_after();

      const int ts = tile_k >> kItemShift;                     // the tile's shard
      const int64_t tile = tile_k & ((1 << kItemShift) - 1);
      const int64_t b = tile * kRows + row;
      const bool valid = b < nblocks;

      // pass 1: sum of squares and extremes of t = H_n x
      f2 ea[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
      float hi[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      float lo[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
      float u[NC][SL];
#pragma unroll 1
      for (int sl = 0; sl < NC; ++sl) {
        load_slice<NC, SL>(tacc, sl, u);
        chunk_butterflies<NC, SL>(u);
        slice_stats<NC, SL>(u, ea, hi, lo);
      }
      const f2 e01 = add2(ea[0], ea[1]), e23 = add2(ea[2], ea[3]);
      const float e = (e01.x + e01.y) + (e23.x + e23.y);   // = n * sum x^2

      // alpha = sqrt(E* / E), E = e / n^2: n sqrt(E*) / sqrt(e), one Newton
      // step, kept in [2^-126, 2^126]; 1 for an all-zero block
      float r = rsqrtf(e);
      r = fmaf(fmaf(-0.5f * e * r, r, 0.5f), r, r);
      float alpha = (e > 0.f) ? clamp_alpha(a.n_sqrtE * r) : 1.0f;
      const float thi = max3(hi[0], hi[1], fmaxf(hi[2], hi[3]));
      const float tlo = min3(lo[0], lo[1], fminf(lo[2], lo[3]));
      const float tmx = fmaxf(thi, -tlo);
      const bool fast = (tmx >= kTrustLo && tmx <= kTrustHi) || tmx == 0.f;
      const bool rescale = !fast && tmx >= kRescaleLo && tmx <= kRescaleHi;
      const bool exact = !fast && !rescale;       // NaN lands here too
      const bool any_rescale = __any_sync(kFullMask, rescale);
      const int kr = rescale ? ilogbf(tmx) : 0;
      const int nkr = -kr, nkr1 = nkr >> 1;       // 2^-k = 2^nkr1 2^(nkr - nkr1), both normal
      const f2 s1{exp2i(nkr1), exp2i(nkr1)}, s2{exp2i(nkr - nkr1), exp2i(nkr - nkr1)};
      if (any_rescale) {
        // the sum of squares of 2^-k t, from tensor memory (the warp reads
        // together)
        const int k = kr;
        f2 eb[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 1
        for (int sl = 0; sl < NC; ++sl) {
          if constexpr (NC > 1) {
            load_slice<NC, SL>(tacc, sl, u);
            chunk_butterflies<NC, SL>(u);
          }
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int i = 0; i < SL; i += 2) {
              const f2 t = mul2(mul2(f2{u[c][i], u[c][i + 1]}, s1), s2);
              eb[(i >> 1) & 3] = fma2(t, t, eb[(i >> 1) & 3]);
            }
        }
        const f2 f01 = add2(eb[0], eb[1]), f23 = add2(eb[2], eb[3]);
        if (rescale) alpha = alpha_scaled(a.n_sqrtE, (f01.x + f01.y) + (f23.x + f23.y), k);
      }
      const float cscale = alpha * a.inv_sqrt_n;             // y = cscale * t
      const float amax = cscale * tmx;
      float sc = (VARIANT == 0)   ? fmaxf(1.0f, amax * (1.0f / QMAX))
                 : (VARIANT == 1) ? (amax > 0.f ? amax * (1.0f / QMAX) : 1.0f)
                                  : a.s_static;
      // code value = gsc * t. Where that factor leaves the fp32 range (a
      // rescaled block of tiny t: ABSMAX's 448 / max |t|, or a tiny E* in
      // STATIC) the warp takes its codes from 2^-k t with the factor times
      // 2^k instead, which stays finite; lanes with k = 0 are unchanged.
      // On the group's last tile the warp's share goes out before the codes,
      // so that the header arrivals overlap them, unless a row of the warp
      // takes the exact path (its alpha and s come after the codes).
      const int nt = __shfl_sync(kFullMask, *n_tiles, 0);
      bool folded = false;
      if (!shared_all && nt >= 0 && k + NG >= nt && !__any_sync(kFullMask, exact && valid)) {
        fold_header(ts, valid, sc);
        __syncwarp();
        if (lane == 0) mbar_arrive(base + S::hdr_ready);
        folded = shared_all = true;
      }
      const float gplain = __fdividef(cscale, sc);
      const bool scaled = __any_sync(kFullMask, rescale && !(gplain <= 0x1.fffffep127f));
      const float gsc = scaled ? __fdividef(ldexpf(cscale, kr), sc) : gplain;

      // pass 2: codes (one slice: the values are still in registers)
      if constexpr (NC == 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(base + S::tempty + 8 * g);
        if (scaled) scale_slice<NC, SL>(u, s1, s2);
        slice_codes<NC, SL, FMT, VARIANT == 2>(u, 0, gsc, staging, row);
      } else {
#pragma unroll 1
        for (int sl = 0; sl < NC; ++sl) {
          load_slice<NC, SL>(tacc, sl, u);
          chunk_butterflies<NC, SL>(u);
          if (scaled) scale_slice<NC, SL>(u, s1, s2);
          slice_codes<NC, SL, FMT, VARIANT == 2>(u, sl, gsc, staging, row);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(base + S::tempty + 8 * g);
      }
      if (exact && valid) {
        const float2 as = exact_block<NB, VARIANT, FMT>(
            a.x + static_cast<int64_t>(ts) * a.shard_elems + b * NB, a.sqrt_nE, a.inv_sqrt_n,
            a.s_static, staging, row);
        alpha = as.x;
        sc = as.y;
      }
      __syncwarp();
      fence_proxy_async_smem();   // codes visible to the tensor store
      group_sync(1 + g);
      if (leader) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
          tma_store_3d(&map_codes, staging + c * kCodeAtomBytes, c * 64,
                       static_cast<int>(tile * kRows), ts);
        bulk_commit();
      }
      if (valid)
        reinterpret_cast<float2*>(a.bundle + static_cast<size_t>(ts) * a.shard_bytes + a.scales_off)[b] =
            make_float2(alpha, sc);
      if (!folded) fold_header(ts, valid, sc);
    }
    // a warp whose last tile did not go out early (or that had none) arrives here
    if (!shared_all) {
      __syncwarp();
      if (lane == 0) mbar_arrive(base + S::hdr_ready);
    }
  }

  // ---- tear-down: free the tensor memory once every store has read the
  // staging buffer (the kernel's end makes the stored codes visible) ----
  tc_fence_before();
  if (warp >= 2 && warp < kSchedWarp && (warp - 2) % 4 == 0 && lane == 0) bulk_wait_read<0>();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Every CTA that shared memory lets onto one SM (228 KB, 1 KB reserved per
// CTA) must find its accumulators in the 512 TMEM columns, or its allocation
// would wait for another CTA to finish.
template <int NB>
constexpr bool fits_sm() {
  return Smem<NB>::bytes <= 232448 &&
         (233472 / (Smem<NB>::bytes + 1024)) * compress_mma_groups(NB) * NB <= 512;
}
static_assert(fits_sm<64>() && fits_sm<128>() && fits_sm<256>(), "shared or tensor memory per SM");

template <int NB, int FMT>
void (*mma_fn(int variant))(CUtensorMap, CUtensorMap, CompressArgs) {
  return variant == 0   ? compress_mma_kernel<NB, 0, FMT>
         : variant == 1 ? compress_mma_kernel<NB, 1, FMT>
                        : compress_mma_kernel<NB, 2, FMT>;
}

template <int FMT>
void (*mma_kernel_fmt(int block, int variant))(CUtensorMap, CUtensorMap, CompressArgs) {
  return block == 64    ? mma_fn<64, FMT>(variant)
         : block == 128 ? mma_fn<128, FMT>(variant)
                        : mma_fn<256, FMT>(variant);
}

void (*mma_kernel(int block, int variant, int fmt))(CUtensorMap, CUtensorMap, CompressArgs) {
  return fmt == 0 ? mma_kernel_fmt<0>(block, variant) : mma_kernel_fmt<1>(block, variant);
}

}  // namespace

EncodeTiled tensor_map_encoder() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

size_t compress_mma_smem_bytes(int block) {
  return block == 64 ? Smem<64>::bytes : block == 128 ? Smem<128>::bytes : Smem<256>::bytes;
}

const void* compress_mma_kernel_ptr(int block, int variant, int fmt) {
  return reinterpret_cast<const void*>(mma_kernel(block, variant, fmt));
}

cudaError_t launch_compress_mma(const CompressArgs& a, int block, int variant, int fmt, int grid_x,
                                int P, cudaStream_t stream) {
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  // x viewed as [P][nblocks][block] bf16; one box = one chunk of 128 blocks.
  CUtensorMap map_x, map_codes;
  const cuuint64_t xdim[3] = {static_cast<cuuint64_t>(block), static_cast<cuuint64_t>(a.nblocks),
                              static_cast<cuuint64_t>(P)};
  const cuuint64_t xstride[2] = {static_cast<cuuint64_t>(block) * 2,
                                 static_cast<cuuint64_t>(a.shard_elems) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kRows), 1};
  const cuuint32_t unit[3] = {1, 1, 1};
  if (encode(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.x), xdim, xstride,
             box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // codes viewed as [P][nblocks][block] bytes with the bundle's shard stride.
  const cuuint64_t cdim[3] = {static_cast<cuuint64_t>(block), static_cast<cuuint64_t>(a.nblocks),
                              static_cast<cuuint64_t>(P)};
  const cuuint64_t cstride[2] = {static_cast<cuuint64_t>(block),
                                 static_cast<cuuint64_t>(a.shard_bytes)};
  if (encode(&map_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.bundle, cdim, cstride, box, unit,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, P);
  cfg.blockDim = dim3(compress_mma_threads(block));
  cfg.dynamicSmemBytes = compress_mma_smem_bytes(block);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mma_kernel(block, variant, fmt), map_x, map_codes, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t compress_mma_fault(unsigned int* bits, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_compress_mma_fault, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_compress_mma_fault, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace taco

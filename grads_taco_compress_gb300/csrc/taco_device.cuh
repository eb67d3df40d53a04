// Device helpers shared by the compress and decompress-reduce kernels.
//
// Element ownership inside one block of NB elements (both kernels):
//   a block is spread over LPB = NB / 64 consecutive lanes of a warp (each
//   lane holds 64 elements); lane j (0 <= j < LPB) of the block holds 8
//   chunks of 8 contiguous elements. Register slot v (0..7) of lane j holds
//   block chunk  j + LPB * (v ^ c),  c = (block index in the warp tile) & 7.
//   The XOR by c makes the 16-byte shared-memory reads of a warp hit distinct
//   banks when the tile was copied contiguously into shared memory.
//   Element index e = 8 * chunk + k therefore has
//     bits 0..2                  -> k        (register index inside a chunk)
//     bits 3 .. 3+log2(LPB)-1    -> j        (lane inside the block)
//     bits 3+log2(LPB) ..        -> v ^ c    (chunk slot)
// The Sylvester Hadamard transform H_NB = H_2 (x) ... (x) H_2 acts on each
// index bit independently: the bits held in registers are transformed in
// registers (packed f32x2 arithmetic), the lane bits with warp shuffles.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "taco.h"

namespace taco {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kCH = 8;                       // chunks of 8 elements per lane
constexpr int kTileElems = 32 * 8 * kCH;     // elements of one warp tile (2048)

// Wall-clock limit of one wait on an mbarrier before the kernel gives up.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;   // 1 s

// Device fault bits (taco_get_fault in taco.h).
constexpr unsigned kFaultCompressWait = 1u;
constexpr unsigned kFaultDecompressWait = 2u;
constexpr unsigned kFaultSelftestWait = 4u;
constexpr unsigned kFaultCompressMmaWait = 8u;
constexpr unsigned kFaultDecompressMmaWait = 16u;

// ------------------------------------------------------- alpha range ----
// alpha = sqrt(E*/E) is stored as an fp32 number and kept inside
// [2^-126, 2^126], where alpha and 1/alpha are both normal fp32 numbers: a
// block whose energy is further than 2^252 from E* is rescaled only part of
// the way, and every decoder can form s / alpha in fp32.
constexpr float kAlphaMin = 0x1p-126f;
constexpr float kAlphaMax = 0x1p126f;
__device__ __forceinline__ float clamp_alpha(float a) { return fminf(fmaxf(a, kAlphaMin), kAlphaMax); }

// A sum of squares accumulated in fp32 is trusted inside [2^-100, 2^100]:
// the squares that fall into fp32's subnormal range then weigh less than
// 2^-40 of it, and neither the sum nor a Hadamard transform of the block
// (|t| <= 256 max|x|) can overflow. Blocks outside are rescaled by a power
// of two first (exactly), which the operator's energy and rotation commute
// with.
constexpr float kEnergyLo = 0x1p-100f;
constexpr float kEnergyHi = 0x1p100f;

// 2^e for -126 <= e <= 127, exactly.
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// alpha for a block whose sum of squares, after scaling the block by 2^-k,
// is e2 (> 0): sqrt(E*/E) = 2^-k * root_E / sqrt(e2), where root_E folds in
// the block's normalisation (sqrt(n E*) for e2 = sum x^2, n sqrt(E*) for
// e2 = sum t^2 of the rotated block, sqrt(E*) for e2 = sum z^2 of a reduced
// one). rsqrt with one Newton step, then 2^-k, then the clamp.
__device__ __forceinline__ float alpha_scaled(float root_E, float e2, int k) {
  float r = rsqrtf(e2);
  r = fmaf(fmaf(-0.5f * e2 * r, r, 0.5f), r, r);
  return clamp_alpha(ldexpf(root_E * r, -k));
}

// ------------------------------------------------------------- f32 pairs ----
// Two fp32 values in one 64-bit register pair, for the packed f32x2 ALU ops.
struct __align__(8) f2 {
  float x, y;
};

__device__ __forceinline__ unsigned long long as_u64(f2 v) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ f2 as_f2(unsigned long long r) {
  f2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(r);
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(r);
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(r);
}
// a * b + c, one rounding per lane
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)), "l"(as_u64(c)));
  return as_f2(r);
}

// ----------------------------------------------------------- bf16 <-> f32 --
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> bf16x2, round to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------- FP8 E4M3 ----
// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448,
// NaN -> 0x7F (the OCP "fn" format). `lo` goes to the low byte.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four fp32 -> four codes in one 32-bit word, element 0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x4_from_f32(float a, float b, float c, float d) {
  return e4m3x2_from_f32(a, b) | (e4m3x2_from_f32(c, d) << 16);
}

// Two E4M3 codes (low byte first) -> two exact fp32 values.
__device__ __forceinline__ f2 e4m3x2_to_f2(uint32_t two_codes) {
  uint32_t h2;
  const uint16_t c = static_cast<uint16_t>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return f2{f.x, f.y};
}

// ------------------------------------------------------ INT8 fallback ----
// Signed-byte codes of the INT8 fallback format: q = round-half-even(y) for
// |y| <= 127 (the scales keep every y in that range). Adding 1.5 * 2^23 to a
// float of magnitude below 2^22 rounds it to an integer k (round to nearest
// even, one fp32 add) and leaves k in the low mantissa bits in two's
// complement, so the low byte is the code.
constexpr float kI8Round = 12582912.0f;   // 1.5 * 2^23

// Four scaled values -> four codes in one word, element 0 in the low byte.
// With CLAMP, values beyond +-127 become +-127 first: the STATIC scale
// bounds |y / s| by 127 only while alpha is not clamped, the other scale
// rules always.
template <bool CLAMP = false>
__device__ __forceinline__ uint32_t i8x4_from_f32(f2 y01, f2 y23);

// Four codes (element 0 in the low byte) -> four exact fp32 values: the
// byte with its sign bit flipped is k + 128 in 0..255; placed under the
// exponent of 1.5 * 2^23 it reads 1.5 * 2^23 + k + 128, and one packed
// subtraction per pair leaves k.
__device__ __forceinline__ void i8x4_to_f32(uint32_t four_codes, f2& v01, f2& v23);

// ------------------------------------------------- shared memory / TMA ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 r;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr));
  return r;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr));
  return r;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes)
               : "memory");
}
// 1-D bulk copy global -> shared (TMA), completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
// 1-D bulk prefetch global -> L2: src 16-byte aligned, bytes a multiple of
// 16. Like the tensor form it returns nothing to the thread, so it may run
// before the preceding grid's writes are visible.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}
// L2 policy for data read once: evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void sts64(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" :: "r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}
// 1-D bulk copy shared -> global (TMA store), tracked in this thread's bulk
// async-group. src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void tma_store_1d(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(dst), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// All but the newest N bulk groups of this thread have finished reading
// their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible (before any global access), and
// let the next grid in the stream begin its launch.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Work of warp w out of W over nblocks blocks, in tiles of BPT blocks:
//   * `rounds` full rounds in grid-stride order (round r, tile r*W + w), so
//     that at any time the warps of the grid stream one contiguous window;
//   * then the blocks left over, split evenly: warp w takes the contiguous
//     range [rlo, rhi) of them, with boundaries on multiples of 4 blocks
//     (every TMA address stays 16-byte aligned), walked in tiles of <= BPT.
// Every block belongs to exactly one tile of one warp.
struct WarpWork {
  int64_t w, W, bpt;
  int64_t rounds;      // full grid-stride rounds
  int64_t rem0;        // first block after the full rounds
  int64_t rlo, rhi;    // this warp's share of the rest, relative to rem0
  int count;           // tiles of this warp

  __device__ __forceinline__ WarpWork(int64_t nblocks, int64_t w_, int64_t W_, int bpt_)
      : w(w_), W(W_), bpt(bpt_) {
    rounds = nblocks / (W * bpt);
    rem0 = rounds * W * bpt;
    const int64_t rest = nblocks - rem0;
    rlo = (rest * w / W) & ~int64_t{3};
    rhi = (w + 1 == W) ? rest : ((rest * (w + 1) / W) & ~int64_t{3});
    if (rhi < rlo) rhi = rlo;
    count = static_cast<int>(rounds + (rhi - rlo + bpt - 1) / bpt);
  }
  // first block and number of blocks of this warp's tile k (0 <= k < count)
  __device__ __forceinline__ void tile(int k, int64_t& b0, int& vb) const {
    if (k < rounds) {
      b0 = (static_cast<int64_t>(k) * W + w) * bpt;
      vb = static_cast<int>(bpt);
    } else {
      b0 = rem0 + rlo + (k - rounds) * bpt;
      const int64_t left = rem0 + rhi - b0;
      vb = static_cast<int>(left < bpt ? left : bpt);
    }
  }
};

// The warp tiles of one CTA as a list that its warps claim in order (a
// shared-memory counter), so that warps the scheduler favours take more of
// them. The list holds the tiles a static split would give the CTA's warps:
// `rounds` full grid-stride rounds (item i: round i / warps, warp slot
// i % warps), then the CTA's even share of the blocks left over, a
// contiguous range on 4-block boundaries cut into tiles of bpt blocks (the
// last may be shorter).
struct CtaWork {
  int64_t W, bpt, c, warps;   // warps of the grid, blocks per tile, CTA, warps per CTA
  int64_t n_full;             // full-round items
  int64_t lo, hi;             // this CTA's share of the rest, absolute blocks
  int64_t total;              // items of this CTA

  __device__ __forceinline__ CtaWork(int64_t nblocks, int64_t c_, int64_t G, int warps_, int bpt_)
      : W(G * warps_), bpt(bpt_), c(c_), warps(warps_) {
    const int64_t rounds = nblocks / (W * bpt);
    const int64_t rem0 = rounds * W * bpt;
    const int64_t rest = nblocks - rem0;
    n_full = rounds * warps;
    lo = rem0 + ((rest * c / G) & ~int64_t{3});
    hi = rem0 + ((c + 1 == G) ? rest : ((rest * (c + 1) / G) & ~int64_t{3}));
    if (hi < lo) hi = lo;
    total = n_full + (hi - lo + bpt - 1) / bpt;
  }
  // first block and number of blocks of item i; false past the end
  __device__ __forceinline__ bool item(int64_t i, int64_t& b0, int& vb) const {
    if (i >= total) return false;
    if (i < n_full) {
      b0 = ((i / warps) * W + c * warps + i % warps) * bpt;
      vb = static_cast<int>(bpt);
    } else {
      b0 = lo + (i - n_full) * bpt;
      const int64_t left = hi - b0;
      vb = static_cast<int>(left < bpt ? left : bpt);
    }
    return true;
  }
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with parity `parity`; false after `limit_ns`
// of wall-clock time without completion.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------- block FWHT -----
// Butterflies on the index bits held in registers (unnormalised H, entries
// +-1). x[q][i] is the f32 pair (elements 2i, 2i+1) of register chunk q.
// `c` is the lane's chunk-slot XOR: register chunk q holds chunk slot q ^ c,
// so for the slot bits the register holding the lower slot of a pair depends
// on c; that butterfly is written as two fmas with a lane-constant sign.
template <int CH>
__device__ __forceinline__ void fwht_in_registers(f2 (&x)[CH][4], int c) {
#pragma unroll
  for (int q = 0; q < CH; ++q) {
    // element bit 0: inside each pair
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = x[q][i].x, b = x[q][i].y;
      x[q][i] = f2{a + b, a - b};
    }
    // element bits 1 and 2: whole pairs
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if ((i & m) == 0) {
          const f2 a = x[q][i], b = x[q][i + m];
          x[q][i] = add2(a, b);
          x[q][i + m] = sub2(a, b);
        }
      }
    }
  }
  // chunk-slot bits
#pragma unroll
  for (int m = 1; m < CH; m <<= 1) {
    const float sg = (c & m) ? -1.0f : 1.0f;
    const f2 sgn{sg, sg}, nsgn{-sg, -sg};
#pragma unroll
    for (int q = 0; q < CH; ++q) {
      if ((q & m) == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const f2 a = x[q][i], b = x[q + m][i];
          x[q][i] = fma2(a, sgn, b);       // c&m == 0: a + b ; else b - a
          x[q + m][i] = fma2(b, nsgn, a);  // c&m == 0: a - b ; else a + b
        }
      }
    }
  }
}

// Butterflies on the lane bits: the lane whose bit is clear keeps a + b, the
// partner keeps a - b (a = the element with the bit clear). One exact
// multiply by +-1 and one rounded add, as in the register stages.
template <int CH, int LPB>
__device__ __forceinline__ void fwht_across_lanes(f2 (&x)[CH][4], int j) {
#pragma unroll
  for (int m = 1; m < LPB; m <<= 1) {
    const float sg = (j & m) ? -1.0f : 1.0f;
    const f2 sgn{sg, sg};
#pragma unroll
    for (int q = 0; q < CH; ++q) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f2 p{__shfl_xor_sync(kFullMask, x[q][i].x, m), __shfl_xor_sync(kFullMask, x[q][i].y, m)};
        x[q][i] = fma2(x[q][i], sgn, p);
      }
    }
  }
}

// Sum / max over the LPB lanes of one block (lanes are consecutive).
template <int LPB>
__device__ __forceinline__ float block_sum(float v) {
#pragma unroll
  for (int m = 1; m < LPB; m <<= 1) v += __shfl_xor_sync(kFullMask, v, m);
  return v;
}

template <int LPB>
__device__ __forceinline__ float block_max(float v) {
#pragma unroll
  for (int m = 1; m < LPB; m <<= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, m));
  return v;
}

// Per-tensor header of one shard, written in the same launch. A CTA folds
// its (max s, count of s > 1) into two running totals in the shard's
// workspace (an atomic max on the float's bits, which order like the values
// because every s is positive and fmaxf drops NaN, and an atomic add), then
// counts its arrival with one acquire-release add. The arrival that
// completes the count takes both totals with one 64-bit exchange that also
// zeroes them, writes the header and resets the counter: two dependent round
// trips to L2 after the last CTA's work.
// Workspace of a shard (16 bytes, zero between calls):
//   [u32 arrivals | u32 tile claims | u32 max-s bits | u32 count]
// (the tensor-core compress lays its own out differently: compress_mma.cu).
__device__ __forceinline__ void write_header(taco_header* hd, int64_t N, int64_t h, int block, int variant,
                                             float target_energy, float q_max, float s_max,
                                             uint32_t n_clamped) {
  hd->N = N;
  hd->h = h;
  hd->block = block;
  hd->variant = variant;
  hd->target_energy = target_energy;
  hd->q_max = q_max;
  hd->s_max = s_max;
  hd->n_clamped = n_clamped;
}
__device__ __forceinline__ void arrive_header(float m, uint32_t n, uint32_t arrivals, uint8_t* ws_shard,
                                              taco_header* hd, int64_t N, int64_t h, int block,
                                              int variant, float target_energy, float q_max) {
  uint32_t* counter = reinterpret_cast<uint32_t*>(ws_shard);
  uint32_t* totals = reinterpret_cast<uint32_t*>(ws_shard + 8);   // 8-byte aligned pair
  if (m > 0.0f)
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(totals), "r"(__float_as_uint(m)) : "memory");
  if (n != 0u)
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(totals + 1), "r"(n) : "memory");
  // the release publishes this CTA's two updates; in the last arrival the
  // acquire orders the exchange below after every other CTA's updates
  uint32_t arrived;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(arrived) : "l"(counter) : "memory");
  if (arrived != arrivals - 1u) return;
  unsigned long long t;
  asm volatile("atom.exch.relaxed.gpu.global.b64 %0, [%1], 0;" : "=l"(t) : "l"(totals) : "memory");
  write_header(hd, N, h, block, variant, target_energy, q_max, __uint_as_float(static_cast<uint32_t>(t)),
               static_cast<uint32_t>(t >> 32));
  // with the exchange, leaves the workspace zero-filled for the next call
  *reinterpret_cast<unsigned long long*>(ws_shard) = 0ull;
}

// One shard per CTA row (gridDim.x CTAs each): every thread brings its
// (max s, count of s > 1), the CTA reduces them and arrives once.
template <int THREADS>
__device__ void finish_header(float part_smax, uint32_t part_cnt, uint8_t* ws_shard,
                              taco_header* hd, int64_t N, int64_t h, int block, int variant,
                              float target_energy, float q_max = 448.0f) {
  constexpr int WARPS = THREADS / 32;
  __shared__ float sh_max[WARPS];
  __shared__ uint32_t sh_cnt[WARPS];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    part_smax = fmaxf(part_smax, __shfl_xor_sync(kFullMask, part_smax, m));
    part_cnt += __shfl_xor_sync(kFullMask, part_cnt, m);
  }
  if (lane == 0) {
    sh_max[warp] = part_smax;
    sh_cnt[warp] = part_cnt;
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  float m = 0.f;
  uint32_t n = 0;
  for (int w = 0; w < WARPS; ++w) {
    m = fmaxf(m, sh_max[w]);
    n += sh_cnt[w];
  }
  arrive_header(m, n, gridDim.x, ws_shard, hd, N, h, block, variant, target_energy, q_max);
}

template <bool CLAMP>
__device__ __forceinline__ uint32_t i8x4_from_f32(f2 y01, f2 y23) {
  if constexpr (CLAMP) {
    y01 = f2{fminf(fmaxf(y01.x, -127.0f), 127.0f), fminf(fmaxf(y01.y, -127.0f), 127.0f)};
    y23 = f2{fminf(fmaxf(y23.x, -127.0f), 127.0f), fminf(fmaxf(y23.y, -127.0f), 127.0f)};
  }
  const f2 m{kI8Round, kI8Round};
  const f2 r01 = add2(y01, m), r23 = add2(y23, m);
  const uint32_t lo = __byte_perm(__float_as_uint(r01.x), __float_as_uint(r01.y), 0x0040);
  const uint32_t hi = __byte_perm(__float_as_uint(r23.x), __float_as_uint(r23.y), 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

__device__ __forceinline__ void i8x4_to_f32(uint32_t four_codes, f2& v01, f2& v23) {
  const uint32_t t = four_codes ^ 0x80808080u;
  const f2 off{kI8Round + 128.0f, kI8Round + 128.0f};
  v01 = sub2(f2{__uint_as_float(__byte_perm(t, 0x4B400000u, 0x7650)),
                __uint_as_float(__byte_perm(t, 0x4B400000u, 0x7651))}, off);
  v23 = sub2(f2{__uint_as_float(__byte_perm(t, 0x4B400000u, 0x7652)),
                __uint_as_float(__byte_perm(t, 0x4B400000u, 0x7653))}, off);
}

// Sum of squares of a lane's 64 values (each scaled by s1 s2 when SCALED),
// in an order that does not depend on the chunk-slot swizzle: each register
// chunk in element order, then a tree that first adds registers q and q ^ 1,
// then those sums at distance 2, then 4. XOR-ing the chunk slots with c maps
// each pair of the tree onto a pair of the same level, and fp32 addition is
// commutative, so the result depends only on the block's values and not on
// where the block sits in its warp tile.
template <bool SCALED>
__device__ __forceinline__ float lane_sum_squares(const f2 (&z)[kCH][4], f2 s1, f2 s2) {
  f2 c[kCH];
#pragma unroll
  for (int q = 0; q < kCH; ++q) {
    f2 v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = SCALED ? mul2(mul2(z[q][r], s1), s2) : z[q][r];
    f2 a = mul2(v[0], v[0]);
    a = fma2(v[1], v[1], a);
    a = fma2(v[2], v[2], a);
    c[q] = fma2(v[3], v[3], a);
  }
#pragma unroll
  for (int m = 1; m < kCH; m <<= 1)
#pragma unroll
    for (int q = 0; q < kCH; ++q)
      if ((q & (2 * m - 1)) == 0) c[q] = add2(c[q], c[q + m]);
  return c[0].x + c[0].y;
}

// Codes of one warp tile's lane (8 chunks of 8 elements, the layout above)
// into shared memory at `base` (byte j + LPB (q ^ cx) * 8 of the block's row):
// code = g * v, with v = 2^-k z when SCALED (s1 s2 = 2^-k), else z.
template <int FMT, int LPB, bool SCALED, bool CLAMP>
__device__ __forceinline__ void store_codes(const f2 (&z)[kCH][4], f2 g2, f2 s1, f2 s2, uint32_t base,
                                            int j, int cx) {
#pragma unroll
  for (int q = 0; q < kCH; ++q) {
    f2 v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = SCALED ? mul2(mul2(z[q][r], s1), s2) : z[q][r];
    const f2 y0 = mul2(v[0], g2), y1 = mul2(v[1], g2), y2 = mul2(v[2], g2), y3 = mul2(v[3], g2);
    uint2 w;
    if constexpr (FMT == 0) {
      w.x = e4m3x4_from_f32(y0.x, y0.y, y1.x, y1.y);
      w.y = e4m3x4_from_f32(y2.x, y2.y, y3.x, y3.y);
    } else {
      w.x = i8x4_from_f32<CLAMP>(y0, y1);
      w.y = i8x4_from_f32<CLAMP>(y2, y3);
    }
    sts64(base + 8 * (j + LPB * (q ^ cx)), w);
  }
}


__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

}  // namespace taco

// Device helpers shared by the compress and decompress-reduce kernels.
//
// Element ownership inside one block of NB elements (both kernels):
//   a block is spread over LPB = NB / (8*CH) consecutive lanes of a warp; lane
//   j (0 <= j < LPB) of the block holds CH chunks of 8 contiguous elements,
//   chunk slot v holding block chunk c = j + LPB*v, i.e. elements 8c .. 8c+7.
//   Element index e = 8c + k therefore has
//     bits 0..2                  -> k  (register index inside a chunk)
//     bits 3 .. 3+log2(LPB)-1    -> j  (lane inside the block)
//     the remaining high bits    -> v  (chunk slot)
// The Sylvester Hadamard transform H_NB = H_2 (x) ... (x) H_2 acts on each
// index bit independently, so the bits held in registers are transformed in
// registers and the lane bits with warp shuffles. Every warp load of a chunk
// slot reads LPB*16 contiguous bytes of each block (whole 32-byte sectors).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace taco {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------- loads ----
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float ld_stream_f32(const float* p) {
  float r;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}

// ----------------------------------------------------------- bf16 <-> f32 --
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack_bf16x8(const uint4& r, float (&x)[8]) {
  x[0] = bf16_lo(r.x); x[1] = bf16_hi(r.x);
  x[2] = bf16_lo(r.y); x[3] = bf16_hi(r.y);
  x[4] = bf16_lo(r.z); x[5] = bf16_hi(r.z);
  x[6] = bf16_lo(r.w); x[7] = bf16_hi(r.w);
}

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
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two_codes) {
  uint32_t h2;
  const uint16_t c = static_cast<uint16_t>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// ---------------------------------------------------------- block FWHT -----
// Butterflies on the index bits held in registers: bits 0..2 inside each
// chunk, then the chunk-slot bits. Unnormalised (H_NB, entries +-1).
template <int CH>
__device__ __forceinline__ void fwht_in_registers(float (&x)[CH][8]) {
#pragma unroll
  for (int v = 0; v < CH; ++v) {
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if ((i & m) == 0) {
          const float a = x[v][i], b = x[v][i + m];
          x[v][i] = a + b;
          x[v][i + m] = a - b;
        }
      }
    }
  }
#pragma unroll
  for (int m = 1; m < CH; m <<= 1) {
#pragma unroll
    for (int v = 0; v < CH; ++v) {
      if ((v & m) == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float a = x[v][i], b = x[v + m][i];
          x[v][i] = a + b;
          x[v + m][i] = a - b;
        }
      }
    }
  }
}

// Butterflies on the lane bits: the lane whose bit is clear keeps a + b, the
// partner keeps a - b (a = the element with the bit clear). One exact
// multiply by +-1 and one rounded add, as in the register stages.
template <int CH, int LPB>
__device__ __forceinline__ void fwht_across_lanes(float (&x)[CH][8], int j) {
#pragma unroll
  for (int m = 1; m < LPB; m <<= 1) {
    const float sgn = (j & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int v = 0; v < CH; ++v) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p = __shfl_xor_sync(kFullMask, x[v][i], m);
        x[v][i] = fmaf(x[v][i], sgn, p);
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

}  // namespace taco

// Elementwise E4M3 codec entry points: the same conversion instructions the
// compress and decompress-reduce kernels use, exposed so that callers (and the
// tests, which sweep every bf16 input) can encode or decode plain arrays.
// Also the self-test of the bounded mbarrier wait that the kernels use.

#include "taco_device.cuh"
#include "taco_launch.h"

namespace taco {

namespace {

__global__ void e4m3_encode_kernel(const float* __restrict__ in, uint8_t* __restrict__ out,
                                   int64_t n) {
  const int64_t i0 = 2 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
  const int64_t step = 2 * static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = i0; i < n; i += step) {
    const float lo = in[i];
    const float hi = (i + 1 < n) ? in[i + 1] : 0.0f;
    const uint32_t two = e4m3x2_from_f32(lo, hi);
    out[i] = static_cast<uint8_t>(two & 0xff);
    if (i + 1 < n) out[i + 1] = static_cast<uint8_t>(two >> 8);
  }
}

__global__ void e4m3_decode_kernel(const uint8_t* __restrict__ in, float* __restrict__ out,
                                   int64_t n) {
  const int64_t i0 = 2 * (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x);
  const int64_t step = 2 * static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = i0; i < n; i += step) {
    const uint32_t lo = in[i];
    const uint32_t hi = (i + 1 < n) ? in[i + 1] : 0u;
    const f2 f = e4m3x2_to_f2(lo | (hi << 8));
    out[i] = f.x;
    if (i + 1 < n) out[i + 1] = f.y;
  }
}

__device__ unsigned int g_selftest_fault;

// One warp waits on an mbarrier that nothing ever completes, with a short
// limit: it must give up, report the time-out and return.
__global__ void selftest_wait_kernel(unsigned long long limit_ns, uint32_t* status) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t addr = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(addr, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool got = mbar_wait(addr, 0, limit_ns);
  const bool all = __all_sync(kFullMask, got);
  if (threadIdx.x == 0) {
    *status = all ? 0u : 1u;
    if (!all) atomicOr(&g_selftest_fault, kFaultSelftestWait);
  }
}

int codec_grid(int64_t n) {
  const int64_t pairs = (n + 1) / 2;
  int64_t g = (pairs + 255) / 256;
  if (g > 4096) g = 4096;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, int64_t n, cudaStream_t st) {
  e4m3_encode_kernel<<<codec_grid(n), 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_decode(const uint8_t* in, float* out, int64_t n, cudaStream_t st) {
  e4m3_decode_kernel<<<codec_grid(n), 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(unsigned long long limit_ns, uint32_t* status, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

cudaError_t selftest_fault(unsigned int* bits, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_selftest_fault, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_selftest_fault, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace taco

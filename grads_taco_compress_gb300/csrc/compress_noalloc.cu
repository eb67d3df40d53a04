// taco_compress_shards_noalloc: compress without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they
// compress: a communication library's progress thread or collective callback
// that must not call cudaMalloc (it can synchronise the device or deadlock
// against work in flight), or a runtime whose memory is owned by an external
// pool. This entry point needs no workspace from them: the arrival counters
// and running totals that write the per-tensor header live in the static
// device array below, which every GPU that loads this library keeps until the
// process exits.

#include <cmath>
#include <mutex>

#include "taco_launch.h"

namespace {

// Room for TACO_NOALLOC_MAX_SHARDS shards of compress workspace (128 B).
constexpr size_t kNoallocScratchBytes =
    static_cast<size_t>(TACO_NOALLOC_MAX_SHARDS) * taco::kWorkspaceShardStride;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_scratch_once[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];

// Device address of the scratch array on the current device. In host code
// `g_noalloc_scratch` is only a host-side stand-in, so the address is looked up
// once per device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_scratch_once[dev], [dev]() {
    void* p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    g_scratch_ptr[dev] = p;
  });
  if (g_scratch_err[dev] != cudaSuccess) return g_scratch_err[dev];
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" taco_status taco_compress_shards_noalloc(const void* x_bf16, int P, int64_t N, int64_t h,
                                                    int block, float target_energy, int variant,
                                                    void* bundle_out, taco_header* headers_out,
                                                    void* stream) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return TACO_ERR_CUDA;   // a lookup, nothing enqueued
  // The checks of taco_compress_shards with the static scratch as the
  // workspace (P beyond its room gives TACO_ERR_WORKSPACE), taken before
  // the scratch clear so that a rejected call enqueues nothing.
  const taco_status st = taco::check_compress_args(x_bf16, P, N, h, block, target_energy, variant,
                                                   bundle_out, headers_out, scratch,
                                                   kNoallocScratchBytes);
  if (st != TACO_OK) return st;
  const size_t need = static_cast<size_t>(P) * taco::kWorkspaceShardStride;
  // The arrival counters must start at zero; the array keeps whatever the
  // previous call (on any stream) left in it.
  if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TACO_ERR_CUDA;
  return taco_compress_shards(x_bf16, P, N, h, block, target_energy, variant, bundle_out,
                              headers_out, scratch, need, stream);
}

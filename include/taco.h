/*
 * taco.h - C ABI of the GB300 (sm_103a) TACO fused compression operator.
 *
 * The operator is the one described for tensor-parallel intermediate tensors
 * in "TACO: Efficient Communication Compression of Intermediate Tensors for
 * Scalable Tensor-Parallel LLM Training" (gist.science Portuguese summary,
 * §2.B.1 "Adaptive Scale-Hadamard transform", §2.B.2 "Dual-Scale
 * quantization", §2.B.3 "fused operator" and "two-shot AllReduce"):
 *
 *   compress, per block of n contiguous elements of a row (n = 64, 128, 256):
 *     E      = mean of x^2 over the block            (raw second moment)
 *     alpha  = sqrt(E* / E)      (1 when E == 0)      (pre-rotation scale),
 *              rounded to fp32 and kept in [2^-126, 2^126], where alpha and
 *              1/alpha are both normal fp32 numbers (a block whose energy is
 *              further than 2^252 from E* is rescaled only part of the way)
 *     y      = (H_n / sqrt(n)) (alpha x)              (Sylvester Hadamard)
 *     s      = max(1, max|y| / 448)                   (post-rotation scale)
 *     q      = E4M3(y / s)   round-to-nearest-even, saturating at +-448
 *   decompress-reduce, over P shards compressed with the same n:
 *     x_hat  = bf16( sum_p (1/alpha_p) (H_n / sqrt(n)) (s_p dec(q_p)) )
 *
 * Conventions of every entry point:
 *   - All buffers are device memory owned by the caller. The library never
 *     allocates, frees or synchronises; work is enqueued on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream) of the device that
 *     is current on the calling thread.
 *   - Arguments are checked on the host before anything is enqueued. On any
 *     error nothing is launched and nothing is written.
 *   - A launch failure is reported as TACO_ERR_CUDA (from cudaGetLastError).
 *   - bf16 tensors are row-major [N, h] with h % n == 0; a block is n
 *     contiguous elements of one row, block b = row * (h/n) + column / n.
 */
#ifndef TACO_H_
#define TACO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum taco_status {
  TACO_OK = 0,
  TACO_ERR_NULL = 1,       /* a required pointer is NULL                       */
  TACO_ERR_SHAPE = 2,      /* N < 0, h <= 0, h % block != 0, or N*h too large  */
  TACO_ERR_BLOCK = 3,      /* block is not 64, 128 or 256                      */
  TACO_ERR_ALIGN = 4,      /* a tensor or bundle pointer is not 16-byte aligned */
  TACO_ERR_ARG = 5,        /* target energy not in (0, 2^120], P out of
                              [1, TACO_MAX_SHARDS], unknown variant            */
  TACO_ERR_CUDA = 6,       /* a CUDA call or launch failed                     */
  TACO_ERR_WORKSPACE = 7   /* workspace NULL or smaller than taco_workspace_bytes */
} taco_status;

/* Dual-scale variants. DUAL is the operator above. ABSMAX replaces the
 * overflow guard by s = max|y| / 448 (1 for an all-zero block); alpha then
 * cancels from the codes. STATIC gives every block of the tensor the same
 * data-independent s = fp32(sqrt(block * E*) / 448): after the energy
 * rescale the rotated block has squared norm block * E*, so no |y| exceeds
 * sqrt(block * E*) and no code saturates (a per-tensor scale in the sense of
 * the euno.news rewrite, Methodology). ABSMAX and STATIC are kept for error
 * studies. */
enum { TACO_VARIANT_DUAL = 0, TACO_VARIANT_ABSMAX = 1, TACO_VARIANT_STATIC = 2 };

#define TACO_MAX_SHARDS 16
#define TACO_Q_MAX 448.0f
#define TACO_ABI_VERSION 1

/* Per-tensor header written by the compress kernel (one per shard).
 * s_max = max over blocks of s (0 for an empty tensor); n_clamped = number of
 * blocks with s > 1. This is the per-tensor part of the dual scale: the
 * "per-tensor scale adapted to the dynamic range" of the euno.news rewrite
 * ("Adaptive Scale-Hadamard Transform" in its Methodology), kept as a
 * summary, not applied to the codes. */
typedef struct taco_header {
  int64_t N;
  int64_t h;
  int32_t block;
  int32_t variant;
  float target_energy;
  float q_max;
  float s_max;
  uint32_t n_clamped;
} taco_header; /* 40 bytes */

/* ---- Shard layout -------------------------------------------------------
 * One compressed tensor ("shard") is one contiguous byte range:
 *   [codes:  N*h bytes, E4M3, row-major][pad to 256]
 *   [scales: N*(h/n) pairs of fp32 (alpha, s), block order][pad to 256]
 * The two scales of a block are adjacent because every reader needs both
 * (TACO pt summary §2.B.2: reconstruction uses alpha_k and s_k together).
 * A bundle is P shards back to back, shard p at p * taco_shard_bytes(...);
 * it is the receive buffer of the ReduceScatter half of the two-shot
 * AllReduce (TACO pt summary, §2.B.3). Both parts start 256-byte aligned
 * relative to the shard start. Return 0 for invalid arguments. */
size_t taco_shard_bytes(int64_t N, int64_t h, int block);
size_t taco_shard_scales_offset(int64_t N, int64_t h, int block);

/* Bytes of device workspace that compress needs for P shards (16 per
 * shard). The workspace holds, per shard, an arrival counter and the running
 * maximum and count used to write the per-tensor header in the same launch;
 * the first shard's slot also holds the counter from which the tensor-core
 * compress hands out tiles of every shard. It must be zero-filled before
 * its first use; each call leaves it zero-filled again. Calls that share a
 * workspace must not overlap on the GPU (use one workspace per stream). */
size_t taco_workspace_bytes(int P);

/* ---- taco_compress ------------------------------------------------------
 * Compress one bf16 tensor x [N, h] (device, 16-byte aligned) into one
 * shard at `shard_out` (device, 16-byte aligned, taco_shard_bytes(N,h,block)
 * bytes) and its header at `header_out` (device, 8-byte aligned).
 *   block          n, one of 64, 128, 256
 *   target_energy  E* in (0, 2^120], the per-element energy of every
 *                  rescaled block (TACO pt summary §2.B.1: each block is
 *                  rescaled to one common energy level); 4096 puts the
 *                  rotated RMS at 64 code units
 *   variant        TACO_VARIANT_DUAL, TACO_VARIANT_ABSMAX or TACO_VARIANT_STATIC
 *   workspace      device memory of taco_workspace_bytes(1) bytes, 16-byte
 *                  aligned, zero before its first use. The pages specify no
 *                  API; this argument is this library's addition to the plain
 *                  compress(x, block, E*) signature, because the per-tensor
 *                  header is written in the same launch (the CTA that
 *                  arrives last reads counters that every CTA updates) and
 *                  the library itself never allocates.
 * Every finite bf16 input is accepted, subnormals and values near the bf16
 * maximum included; no finite input gives a NaN code.
 * N == 0 is valid: no code is written and the header reports s_max = 0. */
taco_status taco_compress(const void* x_bf16, int64_t N, int64_t h, int block,
                          float target_energy, int variant, void* shard_out,
                          taco_header* header_out, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ---- taco_compress_shards -----------------------------------------------
 * The same for P tensors x [P, N, h] (contiguous) in one launch: shard p of
 * the bundle at `bundle_out` (P * taco_shard_bytes bytes) and header p of
 * `headers_out` [P]. 1 <= P <= TACO_MAX_SHARDS. These are the P chunks one
 * rank compresses before the ReduceScatter (TACO pt summary §2.B.3).
 * taco_compress and taco_compress_shards run the tensor-core kernel of
 * taco_compress_shards_mma (below) when a shard holds at most 2^31 - 256
 * blocks, and the CUDA-core kernel of taco_compress_shards_fwht beyond that:
 * the outputs meet the same parity bar either way. */
taco_status taco_compress_shards(const void* x_bf16, int P, int64_t N, int64_t h,
                                 int block, float target_energy, int variant,
                                 void* bundle_out, taco_header* headers_out,
                                 void* workspace, size_t workspace_bytes,
                                 void* stream);

/* ---- taco_compress_shards_fwht ---------------------------------------------
 * taco_compress_shards with the whole rotation as a CUDA-core fast
 * Walsh-Hadamard transform (log2 n butterfly levels in registers and warp
 * shuffles; TACO pt summary §2.B.1 rotates each block by the orthonormal
 * Hadamard matrix): same arguments, layout, headers, workspace and errors,
 * no limit on blocks per shard beyond the shape checks. The energy is summed
 * from x. A code can differ from the tensor-core kernel's by one E4M3 step
 * where the fp32 rotated value differs in its last bits. */
taco_status taco_compress_shards_fwht(const void* x_bf16, int P, int64_t N, int64_t h,
                                      int block, float target_energy, int variant,
                                      void* bundle_out, taco_header* headers_out,
                                      void* workspace, size_t workspace_bytes,
                                      void* stream);

/* ---- taco_compress_shards_mma ----------------------------------------------
 * taco_compress_shards with the Hadamard rotation on the tensor cores
 * (tcgen05, sm_100 family): same arguments, layout, headers, workspace and
 * errors. H_n = H_{n/64} (x) H_64 (Sylvester, TACO pt summary §2.B.1), so
 * every 64-element chunk of a block is multiplied by H_64 as one row of a
 * [128 x 64] x [64 x 64] bf16 product accumulated in fp32, and the
 * log2(n/64) remaining butterfly levels run in registers. The block energy
 * is taken from the rotated block (sum t^2 = n sum x^2). The outputs meet the
 * same parity bar as taco_compress_shards_fwht; a code can differ from that
 * kernel's by one E4M3 step where the fp32 rotated value differs in its last
 * bits. A block whose largest rotated magnitude lies outside [2^-40, 2^56]
 * takes a slower path: its energy is summed again from the rotated values
 * scaled by a power of two, or, for blocks of bf16 subnormals only and
 * blocks near the bf16 maximum whose rotation overflows fp32, the block is
 * redone from x. Extra limit: at most 2^31 - 256 blocks per shard (the tensor
 * copies address rows with 32-bit coordinates), else TACO_ERR_SHAPE.
 * N == 0 writes the headers as taco_compress_shards does. */
taco_status taco_compress_shards_mma(const void* x_bf16, int P, int64_t N, int64_t h,
                                     int block, float target_energy, int variant,
                                     void* bundle_out, taco_header* headers_out,
                                     void* workspace, size_t workspace_bytes,
                                     void* stream);

/* ---- taco_compress_shards_noalloc -----------------------------------------
 * The paper has no counterpart to this entry point: it exists for callers
 * that cannot allocate device memory when they compress (a communication
 * library's progress thread or collective callback, where cudaMalloc may
 * synchronise the device or deadlock against work in flight; a runtime
 * whose memory belongs to an external pool). It is taco_compress_shards
 * without the workspace argument: the counters and running totals live in
 * a static device array of the library (TACO_NOALLOC_MAX_SHARDS * 16 = 128
 * bytes), which every GPU that loads the library holds until the process
 * exits. The caller still passes x, the bundle and the headers.
 *   - P > TACO_NOALLOC_MAX_SHARDS returns TACO_ERR_WORKSPACE (the request does
 *     not fit the static scratch); other errors as taco_compress_shards, and a
 *     rejected call enqueues nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Each call clears the counters it uses with cudaMemsetAsync on `stream`
 *     and then launches the compress kernel; it allocates nothing.
 *   - All calls share the one array, so calls that overlap on the GPU (other
 *     streams, other threads) race on it: order them. */
#define TACO_NOALLOC_MAX_SHARDS 8
taco_status taco_compress_shards_noalloc(const void* x_bf16, int P, int64_t N, int64_t h,
                                         int block, float target_energy, int variant,
                                         void* bundle_out, taco_header* headers_out,
                                         void* stream);

/* ---- taco_decompress_reduce ---------------------------------------------
 * Reconstruct and sum P shards of one bundle (device, 16-byte aligned, the
 * layout above, all compressed from [N, h] tensors with the same block)
 * into bf16 out [N, h] (device, 16-byte aligned). The P reconstructions are
 * summed in fp32 in the rotated domain and rotated back once (the rotation is
 * linear and shared by all shards), then rounded to bf16 once. This is the
 * reconstruction of TACO pt summary §2.B.2 fused with the reduce of the
 * ReduceScatter step of §2.B.3. 1 <= P <= TACO_MAX_SHARDS. N == 0 is valid
 * and launches nothing. `out` must not overlap the bundle. */
taco_status taco_decompress_reduce(const void* bundle, int P, int64_t N, int64_t h,
                                   int block, void* out_bf16, void* stream);

/* ---- taco_decompress_reduce_mma[_ptrs] ------------------------------------
 * taco_decompress_reduce[_ptrs] with the inverse rotation on the tensor
 * cores (tcgen05, E4M3 operands): same arguments, layout and errors, for
 * block 64 or 128 (block 256 returns TACO_ERR_BLOCK). By linearity
 * x_hat = sum_p (s_p / (alpha_p sqrt(n))) H_n q_p (TACO pt summary §2.B.2,
 * reduce of §2.B.3); each 64-code chunk of each shard is multiplied by H_64
 * as it arrives, exactly in fp32, the scaled sum over shards and the
 * remaining butterfly levels run in registers, one bf16 rounding at the end.
 * The output meets the reconstruction bar of taco_decompress_reduce; the two
 * entries sum in different orders, so single bf16 results may differ by one
 * unit in the last place. At most 2^31 - 256 blocks per shard. */
taco_status taco_decompress_reduce_mma(const void* bundle, int P, int64_t N, int64_t h,
                                       int block, void* out_bf16, void* stream);
taco_status taco_decompress_reduce_mma_ptrs(const void* const* shards, int P, int64_t N,
                                            int64_t h, int block, void* out_bf16, void* stream);

/* ---- INT8 fallback format -------------------------------------------------
 * TACO pt summary §5 ("Agnóstico de Hardware"): the framework degrades to
 * INT8 on hardware without FP8 support. The pages define no INT8 format
 * beyond the uniform steps of §2.A; these entries take the plainest reading:
 * every step of the operator as above, with the code of a rotated value y
 * being q = round-half-to-even(y / s) as a signed byte (two's complement,
 * never -128) and Q_max = 127 in place of 448 in the scale rules (DUAL:
 * s = max(1, max|y| / 127); ABSMAX: s = max|y| / 127; STATIC:
 * s = sqrt(block * E*) / 127). The headers report q_max = 127. Same shard
 * layout, arguments, workspace and errors as taco_compress_shards_mma /
 * taco_decompress_reduce; the rotation runs on the tensor cores. A bundle
 * must be decompressed with the entry of its format. */
taco_status taco_compress_shards_int8(const void* x_bf16, int P, int64_t N, int64_t h,
                                      int block, float target_energy, int variant,
                                      void* bundle_out, taco_header* headers_out,
                                      void* workspace, size_t workspace_bytes,
                                      void* stream);
taco_status taco_decompress_reduce_int8(const void* bundle, int P, int64_t N, int64_t h,
                                        int block, void* out_bf16, void* stream);
/* The AllGather side and the step between the two halves of the two-shot
 * AllReduce in the INT8 format: taco_reduce_recompress_ptrs and
 * taco_decompress_shards_ptrs with INT8 codes in and out (q_max 127 in the
 * written header). */
taco_status taco_reduce_recompress_int8_ptrs(const void* const* shards, int P, int64_t N,
                                             int64_t h, int block, float target_energy,
                                             int variant, void* shard_out,
                                             taco_header* header_out, void* out_bf16,
                                             void* workspace, size_t workspace_bytes,
                                             void* stream);
taco_status taco_decompress_shards_int8_ptrs(const void* const* shards, int P, int64_t N,
                                             int64_t h, int block, void* out_bf16, void* stream);

/* ---- taco_reduce_recompress_batched_ptrs --------------------------------
 * Y independent reduce-recompress operations in one launch: the step between
 * the ReduceScatter and the AllGather (TACO pt summary §2.B.3) for Y
 * destinations at once. Reduction y sums shards[y*P .. y*P+P-1] (host array
 * of Y*P device pointers, 1 <= Y*P <= TACO_MAX_SHARDS) and writes shard y of
 * `shards_out` (Y consecutive shards of taco_shard_bytes, device, 16-byte
 * aligned) and headers_out[y]; the workspace holds Y shard workspaces
 * (taco_workspace_bytes(Y)). code_format: TACO_FORMAT_E4M3 or
 * TACO_FORMAT_INT8 (codes in and out). No bf16 side output. Otherwise as
 * taco_reduce_recompress_ptrs. */
enum { TACO_FORMAT_E4M3 = 0, TACO_FORMAT_INT8 = 1 };
taco_status taco_reduce_recompress_batched_ptrs(const void* const* shards, int Y, int P, int64_t N,
                                                int64_t h, int block, float target_energy,
                                                int variant, int code_format, void* shards_out,
                                                taco_header* headers_out, void* workspace,
                                                size_t workspace_bytes, void* stream);

/* ---- taco_decompress_reduce_ptrs ----------------------------------------
 * As taco_decompress_reduce, with the P shards in P separate buffers
 * (`shards[p]` a device pointer to one shard, 16-byte aligned; `shards` itself
 * is a host array of P pointers, read before the call returns). This is the
 * form a receive step that lands each peer's chunk in its own buffer uses. */
taco_status taco_decompress_reduce_ptrs(const void* const* shards, int P, int64_t N,
                                        int64_t h, int block, void* out_bf16,
                                        void* stream);

/* ---- taco_decompress_shards ---------------------------------------------
 * Reconstruct each of the P shards of `bundle` on its own (no sum) into
 * out_bf16 [P][N][h]: shard p to rows p*N .. p*N+N-1. This is the receive
 * side of the AllGather half of the two-shot AllReduce (TACO pt summary
 * §2.B.3), where every rank expands the P reduced chunks into the full
 * tensor; the reconstruction is that of §2.B.2, the same arithmetic as
 * taco_decompress_reduce with P = 1 (bit-identical output). One launch.
 * N == 0 launches nothing. */
taco_status taco_decompress_shards(const void* bundle, int P, int64_t N, int64_t h, int block,
                                   void* out_bf16, void* stream);

/* The same with the shards in separate buffers (host array of P pointers). */
taco_status taco_decompress_shards_ptrs(const void* const* shards, int P, int64_t N, int64_t h,
                                        int block, void* out_bf16, void* stream);

/* ---- taco_reduce_recompress ---------------------------------------------
 * The reduced chunk compressed again for the AllGather half of the two-shot
 * AllReduce (TACO pt summary §2.B.3: compression around ReduceScatter +
 * AllGather), fused with the reduce: the P shards of `bundle` (as for
 * taco_decompress_reduce) are summed and the sum x_hat is compressed into
 * one shard at `shard_out` with its header at `header_out`, with the same
 * block, target energy and variant rules as taco_compress. x_hat is
 * compressed as computed, without rounding it to bf16 first. Because the
 * rotation is shared and orthogonal, this needs no Hadamard transform on the
 * device: the rotated sum is already at hand. If `out_bf16` is not NULL the
 * bf16 sum [N, h] is written there as well (bit-identical to
 * taco_decompress_reduce). `workspace`: at least taco_workspace_bytes(1)
 * zero-filled bytes, as for compress. No output may overlap an input. */
taco_status taco_reduce_recompress(const void* bundle, int P, int64_t N, int64_t h, int block,
                                   float target_energy, int variant, void* shard_out,
                                   taco_header* header_out, void* out_bf16, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* The same with the P shards in separate buffers (`shards`: host array of P
 * device pointers, read before the call returns). */
taco_status taco_reduce_recompress_ptrs(const void* const* shards, int P, int64_t N, int64_t h,
                                        int block, float target_energy, int variant,
                                        void* shard_out, taco_header* header_out, void* out_bf16,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* ---- E4M3 codec ----------------------------------------------------------
 * Elementwise conversions with the instructions the operator's kernels use
 * (TACO pt summary §2.A: FP8 E4M3 instead of INT8). `in` and `out` are device
 * arrays of n elements; n == 0 launches nothing.
 *   taco_e4m3_encode_f32: fp32 -> E4M3 code, round to nearest even, |v| > 448
 *                         and +-inf saturate to +-448, NaN -> 0x7F.
 *   taco_e4m3_decode_f32: E4M3 code -> its exact fp32 value (0x7F/0xFF: NaN). */
taco_status taco_e4m3_encode_f32(const float* in, uint8_t* out, int64_t n, void* stream);
taco_status taco_e4m3_decode_f32(const uint8_t* in, float* out, int64_t n, void* stream);

/* ---- Device faults ---------------------------------------------------------
 * The kernels wait on shared-memory barriers for their bulk copies; each wait
 * gives up after one second of wall-clock time, sets a bit in a device-side
 * fault word of the library, lets the copies still in flight land (again
 * bounded) and returns, so that a fault never hangs the GPU. Bits:
 *   TACO_FAULT_COMPRESS_WAIT, TACO_FAULT_DECOMPRESS_WAIT, TACO_FAULT_SELFTEST_WAIT,
 *   TACO_FAULT_COMPRESS_MMA_WAIT (taco_compress_shards_mma: a wait on a copy,
 *   an MMA or the epilogue gave up; the CTA drains its MMAs and copies and
 *   frees its tensor memory before it returns), TACO_FAULT_DECOMPRESS_MMA_WAIT
 *   (the same for taco_decompress_reduce_mma).
 * taco_get_fault reads (and with clear != 0 resets) the word of the current
 * device; it synchronises with the device. */
#define TACO_FAULT_COMPRESS_WAIT 1u
#define TACO_FAULT_DECOMPRESS_WAIT 2u
#define TACO_FAULT_SELFTEST_WAIT 4u
#define TACO_FAULT_COMPRESS_MMA_WAIT 8u
#define TACO_FAULT_DECOMPRESS_MMA_WAIT 16u
taco_status taco_get_fault(uint32_t* bits, int clear);

/* Self-test of that time-out path: one warp waits on a barrier that nothing
 * completes, for limit_ns (1 .. 2e9) nanoseconds, then writes 1 to
 * *status_dev (a device word) and sets TACO_FAULT_SELFTEST_WAIT; 0 would
 * mean the wait completed, which it cannot. */
taco_status taco_selftest_wait_timeout(uint64_t limit_ns, uint32_t* status_dev, void* stream);

/* Human-readable name of a status code (static storage). */
const char* taco_status_string(taco_status status);

/* TACO_ABI_VERSION of the loaded library. */
int taco_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TACO_H_ */

"""Plain CPU oracle of the TACO compress / decompress-reduce operator.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute this module: it is imported by ``tests/``, by ``__graft_entry__.smoke()``
(to check one small GPU call) and by the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``. It shares no code with the CUDA library.

What it computes, and where the method is stated
------------------------------------------------
Sources are the pages on "TACO: Efficient Communication Compression of
Intermediate Tensors for Scalable Tensor-Parallel LLM Training":

  [PT]  gist.science Portuguese technical summary (paper 2604.24088)
  [DE]  gist.science German lay summary (same paper)
  [ZH]  euno.news Chinese rewrite of the arXiv abstract (same paper)

Compress, per block of ``n`` contiguous elements of one row
(  [PT] §2.B.1 "Adaptive Scale-Hadamard transform (ASH)",
   [PT] §2.B.2 "Dual-Scale quantization (DS)",
   [PT] §2.A   "Why FP8?" -> E4M3 )
  1. energy   E_k = raw (uncentred) second moment of the block, mean over n
  2. alpha_k  = sqrt(E* / E_k), rounded once to fp32 and kept inside
              [2^-126, 2^126] (alpha_k = 1 if E_k = 0)
  3. rotate   y = (H_n / sqrt(n)) (alpha_k x), Sylvester H_n, rounded to fp32
  4. s_k      = max(1, max_i |y_i| / Q_max), Q_max = 448, rounded to fp32
  5. q_i      = E4M3 round-to-nearest-even with saturation of fp32(y_i / s_k)
  6. per-tensor header: s_max = max_k s_k, n_clamped = #{k : s_k > 1}
Decompress-reduce ([PT] §2.B.2 "Reconstruction"; the reduce of the
ReduceScatter half of the two-shot AllReduce, [PT] §2.B.3):
  x_hat = bf16_RNE( sum_p (1/alpha_p) (H_n^T / sqrt(n)) (s_p * dec(q_p)) )
in fp64, inverting each shard on its own and summing: the plain definition.
Reduce-recompress (the reduced chunk compressed again for the AllGather,
[PT] §2.B.3): the compress steps applied to the fp64 x_hat above, before
any rounding to bf16.
INT8 fallback ([PT] §5 "Agnóstico de Hardware": the framework degrades to
INT8 on hardware without FP8): every step above with the code format
replaced, q_i = round-half-even(y_i / s_k) as a signed byte, Q_max = 127 in
the scale rules, decoded as the integer itself. The pages give no more than
"INT8"; this symmetric uniform reading is the plainest one.

Readings taken where the pages are silent (each one is a choice):
  * dual scale: alpha_k sets the block energy before rotation (the
    anti-underflow role of [DE] §3), s_k = max(1, amax/Q_max) is the overflow
    guard that makes the rotated values fit Q_max ([PT] §2.B.2). Variant
    ABSMAX (s_k = amax/Q_max for amax > 0, else 1) is kept for comparison; in
    it alpha_k cancels from the codes. Variant STATIC (one data-independent
    s = sqrt(n E*)/Q_max for every block of the tensor, a per-tensor scale in
    the sense of [ZH]) is kept for error studies: after the energy rescale
    ||y||_2^2 = n E*, so by Cauchy-Schwarz |y_i| <= sqrt(n E*) and no code
    ever saturates.
  * "energy" is the mean of squares (E* is per element), uncentred.
  * Hadamard: Sylvester natural order, orthonormal scaling 1/sqrt(n), no sign
    flips. The same n-element blocks carry alpha, the rotation and s.
  * E4M3 is the OCP "fn" format: bias 7, 3 mantissa bits, subnormals
    m * 2^-9, largest finite 448 (0x7E), 0x7F/0xFF are NaN, no infinities.
    Rounding: nearest, ties to the even code; |v| > 448 and +-inf saturate to
    +-448; NaN -> 0x7F; the sign is kept (values that round to zero from
    below give 0x80).
  * The value handed to the E4M3 rounding is an fp32 number on both the
    oracle and the GPU path, so both take that integer decision in fp32.
  * alpha is stored as an fp32 number, and the pages put no magnitude limit
    on a block, so the rescale has to be defined where sqrt(E*/E_k) does not
    fit: alpha_k is sqrt(E*/E_k) rounded to fp32 and then clamped to
    [2^-126, 2^126], the range in which both alpha_k and 1/alpha_k are
    normal fp32 numbers. A block whose energy is more than 2^252 away from
    E* (for E* = 4096: an RMS below 2^-120, i.e. bf16 subnormals and the
    smallest normals, or above 2^132, which bf16 cannot hold) is rescaled
    only part of the way; its codes still decode with the alpha that was
    applied, and no finite input gives a NaN or infinite code, alpha or s.
    Inside the range the operator is exactly equivariant under powers of
    two: compress(2^k x) has the codes and s of compress(x) and alpha
    scaled by exactly 2^-k.

Parity pins live in ``tests/test_oracle_pins.py`` (Hadamard against its
closed form and scipy, the E4M3 codec against torch's float8_e4m3fn and the
format's printed points, bf16 rounding against torch, energy invariant,
spike / constant / zero blocks in closed form). The choice of dual-scale
variant and of E* itself cannot be pinned by the pages: parity unpinned for
those two readings.
"""

from __future__ import annotations

import math

import numpy as np

Q_MAX = 448.0
Q_MAX_INT8 = 127.0
FORMAT_E4M3 = 0
FORMAT_INT8 = 1
DEFAULT_TARGET_ENERGY = 4096.0
ALPHA_MIN = 2.0 ** -126        # alpha and 1/alpha both normal fp32 numbers
ALPHA_MAX = 2.0 ** 126
VARIANT_DUAL = 0
VARIANT_ABSMAX = 1
VARIANT_STATIC = 2
VARIANTS = (VARIANT_DUAL, VARIANT_ABSMAX, VARIANT_STATIC)
BLOCK_SIZES = (64, 128, 256)


# --------------------------------------------------------------------------
# Sylvester Hadamard matrix ([PT] §2.B.1: orthogonal Hadamard rotation)
# --------------------------------------------------------------------------
def sylvester_hadamard(n: int) -> np.ndarray:
    """H_1 = [1];  H_2m = [[H_m, H_m], [H_m, -H_m]].  Integer +-1 entries."""
    if n < 1 or n & (n - 1):
        raise ValueError("Hadamard order must be a power of two")
    h = np.ones((1, 1), dtype=np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


# --------------------------------------------------------------------------
# FP8 E4M3 ("fn" variant) codec ([PT] §2.A: E4M3 chosen over INT8)
# --------------------------------------------------------------------------
def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 codes, read from the bit fields."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        man_field = code & 0x7
        if exp_field == 0xF and man_field == 0x7:
            vals[code] = np.nan
        elif exp_field == 0:
            vals[code] = sign * man_field * 2.0 ** -9          # subnormal
        else:
            vals[code] = sign * (1.0 + man_field / 8.0) * 2.0 ** (exp_field - 7)
    return vals


_E4M3_TABLE = e4m3_decode_table()
# The 127 non-negative finite values, codes 0x00..0x7E, in increasing order.
_E4M3_NONNEG = _E4M3_TABLE[:127].copy()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Round fp32 values to E4M3 codes by nearest-value search.

    The nearest of the 127 non-negative finite magnitudes is taken; on a tie
    the code with a zero last mantissa bit (an even code) wins. Magnitudes
    above 448 (and infinities) give 448. NaN gives 0x7F. The sign bit is the
    sign bit of the input, zeros included.
    """
    v32 = np.asarray(v, dtype=np.float32)
    mag = np.abs(v32).astype(np.float64)
    nan = np.isnan(v32)
    mag_safe = np.where(nan, 0.0, mag)
    hi = np.searchsorted(_E4M3_NONNEG, mag_safe, side="left")   # first value >= mag
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag_safe - _E4M3_NONNEG[lo]
    d_hi = _E4M3_NONNEG[hi] - mag_safe
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag_safe >= Q_MAX, 126, code)                 # saturate
    sign = np.signbit(v32).astype(np.int64) << 7
    out = (code | sign).astype(np.uint8)
    out[nan] = 0x7F
    return out


# --------------------------------------------------------------------------
# INT8 codec of the fallback format ([PT] §5; uniform steps, [PT] §2.A)
# --------------------------------------------------------------------------
def int8_encode(v) -> np.ndarray:
    """fp32 values -> signed bytes (as uint8 bit patterns).

    Round to the nearest integer, ties to even, then clamp to [-127, 127]
    (symmetric: -128 is never produced). NaN gives 0.
    """
    v32 = np.asarray(v, dtype=np.float32).astype(np.float64)
    q = np.rint(np.where(np.isnan(v32), 0.0, v32))
    q = np.clip(q, -Q_MAX_INT8, Q_MAX_INT8)
    return q.astype(np.int64).astype(np.int8).view(np.uint8)


def int8_decode(codes: np.ndarray) -> np.ndarray:
    return np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.float64)


def q_max(fmt: int) -> float:
    if fmt == FORMAT_E4M3:
        return Q_MAX
    if fmt == FORMAT_INT8:
        return Q_MAX_INT8
    raise ValueError("unknown code format")


def encode(fmt: int, v) -> np.ndarray:
    return e4m3_encode(v) if fmt == FORMAT_E4M3 else int8_encode(v)


def decode(fmt: int, codes) -> np.ndarray:
    return e4m3_decode(codes) if fmt == FORMAT_E4M3 else int8_decode(codes)


# --------------------------------------------------------------------------
# bfloat16 helpers (inputs are bf16; the reduce writes bf16)
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits and the fp32 exponent range; below 2^-126
    the spacing stays 2^-133 (subnormals). One rounding, straight from fp64.
    Results above the largest finite bf16 become +-inf.
    """
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    finite = np.isfinite(v) & (v != 0)
    _, e = np.frexp(v[finite])                 # |v| = m 2^e, 0.5 <= m < 1
    q = np.maximum(e - 8, -133)                # spacing of bf16 values there
    out[finite] = np.ldexp(np.rint(np.ldexp(v[finite], -q)), q)  # rint: ties even
    big = np.abs(out) >= 2.0 ** 128
    out[big] = np.copysign(np.inf, out[big])
    return out


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round to bf16 (as above) and return the uint16 bit patterns."""
    r = round_to_bf16(v).astype(np.float32)    # exact: bf16 is a subset of fp32
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# Compress
# --------------------------------------------------------------------------
def _check_shape(h: int, block: int) -> None:
    if block not in BLOCK_SIZES:
        raise ValueError(f"block must be one of {BLOCK_SIZES}")
    if h % block:
        raise ValueError("hidden size must be a multiple of the block size")


def compress_stages(x_bits: np.ndarray, block: int,
                    target_energy: float = DEFAULT_TARGET_ENERGY,
                    variant: int = VARIANT_DUAL, fmt: int = FORMAT_E4M3) -> dict:
    """Compress a bf16 [N, h] tensor, returning every intermediate.

    ``x_bits`` holds bf16 bit patterns (uint16). Returned arrays, with
    K = h / block: ``energy`` f64 [N,K], ``alpha`` f32 [N,K], ``y`` f32
    [N,K,n], ``amax`` f64 [N,K], ``s`` f32 [N,K], ``codes`` u8 [N,h] and the
    per-tensor ``header`` dict.
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    return compress_values_stages(bf16_bits_to_f64(x_bits), block, target_energy, variant, fmt)


def compress_values_stages(x_values: np.ndarray, block: int,
                           target_energy: float = DEFAULT_TARGET_ENERGY,
                           variant: int = VARIANT_DUAL, fmt: int = FORMAT_E4M3) -> dict:
    """The same steps on real values [N, h] (float64) instead of bf16 inputs.

    Used for the compression of a reduced tensor that never went through a
    bf16 buffer (the ReduceScatter output recompressed for the AllGather,
    TACO pt summary §2.B.3).
    """
    x_values = np.asarray(x_values, dtype=np.float64)
    N, h = x_values.shape
    n = block
    _check_shape(h, n)
    if variant not in VARIANTS:
        raise ValueError("unknown variant")
    qm = q_max(fmt)
    K = h // n
    x = x_values.reshape(N, K, n)

    # 1. block energy: raw second moment, mean over the block ([PT] §2.B.1)
    energy = np.sum(x * x, axis=-1) / n

    # 2. pre-rotation scale alpha_k: energy of alpha_k x equals E* ([PT] §2.B.2),
    #    as far as an fp32 alpha whose reciprocal is a normal fp32 number allows
    alpha = np.ones((N, K), dtype=np.float32)
    nz = energy > 0
    alpha[nz] = np.clip(np.sqrt(target_energy / energy[nz]), ALPHA_MIN, ALPHA_MAX).astype(np.float32)

    # 3. orthogonal Hadamard rotation of the rescaled block ([PT] §2.B.1)
    H = sylvester_hadamard(n).astype(np.float64)
    scaled = alpha.astype(np.float64)[..., None] * x
    y = ((scaled @ H.T) / math.sqrt(n)).astype(np.float32)

    # 4. post-rotation scale s_k: fit the rotated block into Q_max ([PT] §2.B.2)
    amax = np.max(np.abs(y.astype(np.float64)), axis=-1)
    if variant == VARIANT_DUAL:
        s = np.maximum(1.0, amax / qm).astype(np.float32)
    elif variant == VARIANT_ABSMAX:
        s = np.where(amax > 0, amax / qm, 1.0).astype(np.float32)
    else:
        # one scale for the whole tensor, fixed by E*, n and Q_max alone
        s = np.full((N, K), np.float32(static_scale(n, target_energy, fmt)), dtype=np.float32)

    # 5. FP8 E4M3 codes of y / s_k (the value rounded is an fp32 number)
    ratio = (y.astype(np.float64) / s.astype(np.float64)[..., None]).astype(np.float32)
    codes = encode(fmt, ratio).reshape(N, h)

    # 6. per-tensor header
    header = {
        "N": N, "h": h, "block": n, "variant": variant,
        "target_energy": float(np.float32(target_energy)), "q_max": qm,
        "s_max": float(s.max()) if s.size else 0.0,
        "n_clamped": int(np.count_nonzero(s > 1.0)),
    }
    return {"energy": energy, "alpha": alpha, "y": y, "amax": amax, "s": s,
            "codes": codes, "header": header}


def static_scale(block: int, target_energy: float = DEFAULT_TARGET_ENERGY,
                 fmt: int = FORMAT_E4M3) -> float:
    """fp32(sqrt(n E*) / Q_max): the STATIC variant's scale of every block."""
    return float(np.float32(math.sqrt(block * float(target_energy)) / q_max(fmt)))


def compress(x_bits: np.ndarray, block: int,
             target_energy: float = DEFAULT_TARGET_ENERGY,
             variant: int = VARIANT_DUAL, fmt: int = FORMAT_E4M3):
    """(codes u8 [N,h], alpha f32 [N,K], s f32 [N,K], header dict)."""
    st = compress_stages(x_bits, block, target_energy, variant, fmt)
    return st["codes"], st["alpha"], st["s"], st["header"]


# --------------------------------------------------------------------------
# Decompress-reduce
# --------------------------------------------------------------------------
def decompress_one_f64(codes: np.ndarray, alpha: np.ndarray, s: np.ndarray,
                       block: int, fmt: int = FORMAT_E4M3) -> np.ndarray:
    """Reconstruct one shard in fp64: undo s, the rotation, then alpha."""
    codes = np.asarray(codes, dtype=np.uint8)
    N, h = codes.shape
    n = block
    _check_shape(h, n)
    K = h // n
    q = decode(fmt, codes).reshape(N, K, n)
    w = np.asarray(s, dtype=np.float32).astype(np.float64)[..., None] * q
    H = sylvester_hadamard(n).astype(np.float64)
    # inverse of the orthonormal rotation H/sqrt(n) is its transpose
    u = (w @ H) / math.sqrt(n)          # row form of (H^T / sqrt(n)) w
    xr = u / np.asarray(alpha, dtype=np.float32).astype(np.float64)[..., None]
    return xr.reshape(N, h)


def decompress_reduce_f64(codes: np.ndarray, alpha: np.ndarray, s: np.ndarray,
                          block: int, fmt: int = FORMAT_E4M3) -> np.ndarray:
    """Sum over the P shards of the fp64 reconstructions (before rounding).

    ``codes`` u8 [P,N,h], ``alpha`` and ``s`` f32 [P,N,K].
    """
    codes = np.asarray(codes, dtype=np.uint8)
    P = codes.shape[0]
    total = np.zeros(codes.shape[1:], dtype=np.float64)
    for p in range(P):
        total += decompress_one_f64(codes[p], alpha[p], s[p], block, fmt)
    return total


def decompress_reduce(codes: np.ndarray, alpha: np.ndarray, s: np.ndarray,
                      block: int, fmt: int = FORMAT_E4M3) -> np.ndarray:
    """bf16 bit patterns [N,h] of the reduced reconstruction (one RNE)."""
    return f64_to_bf16_bits(decompress_reduce_f64(codes, alpha, s, block, fmt))


# --------------------------------------------------------------------------
# Reduce then recompress (the step between ReduceScatter and AllGather)
# --------------------------------------------------------------------------
def reduce_recompress(codes: np.ndarray, alpha: np.ndarray, s: np.ndarray, block: int,
                      target_energy: float = DEFAULT_TARGET_ENERGY,
                      variant: int = VARIANT_DUAL, fmt: int = FORMAT_E4M3):
    """Compress the sum of the P reconstructions without rounding it to bf16.

    In the two-shot AllReduce ([PT] §2.B.3) each rank reduces the P chunks
    it received and compresses the reduced chunk again for the AllGather.
    The plain definition: x_hat = decompress_reduce_f64(...) in fp64, then
    the compress steps on those values. Returns (codes, alpha, s, header).
    """
    x_hat = decompress_reduce_f64(codes, alpha, s, block, fmt)
    st = compress_values_stages(x_hat, block, target_energy, variant, fmt)
    return st["codes"], st["alpha"], st["s"], st["header"]


# --------------------------------------------------------------------------
# Wire size ([PT] §5 / [ZH] results: FP8 codes roughly halve TP traffic)
# --------------------------------------------------------------------------
def wire_bytes_per_element(block: int) -> float:
    """One code byte plus two fp32 scales per block of ``block`` elements."""
    return 1.0 + 8.0 / block

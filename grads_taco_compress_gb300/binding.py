"""Thin Python binding of libtaco (the C ABI in include/taco.h).

Argument marshalling only: every step of the operator runs in the CUDA
kernels of libtaco. torch is used for device memory and streams. When the
library has not been built this module raises on first use; there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import pathlib

import numpy as np
import torch

LIB_PATH = pathlib.Path(__file__).resolve().parent / "lib" / "libtaco.so"

TACO_OK = 0
STATUS_NAMES = {0: "TACO_OK", 1: "TACO_ERR_NULL", 2: "TACO_ERR_SHAPE", 3: "TACO_ERR_BLOCK",
                4: "TACO_ERR_ALIGN", 5: "TACO_ERR_ARG", 6: "TACO_ERR_CUDA",
                7: "TACO_ERR_WORKSPACE"}
VARIANT_DUAL = 0
VARIANT_ABSMAX = 1
VARIANT_STATIC = 2
FORMAT_E4M3 = 0
FORMAT_INT8 = 1
MAX_SHARDS = 16
HEADER_BYTES = 40
DEFAULT_TARGET_ENERGY = 4096.0

#: struct taco_header as a numpy record
HEADER_DTYPE = np.dtype([("N", "<i8"), ("h", "<i8"), ("block", "<i4"), ("variant", "<i4"),
                         ("target_energy", "<f4"), ("q_max", "<f4"), ("s_max", "<f4"),
                         ("n_clamped", "<u4")])
assert HEADER_DTYPE.itemsize == HEADER_BYTES

#: every symbol include/taco.h declares
EXPORTED_SYMBOLS = (
    "taco_shard_bytes", "taco_shard_scales_offset",
    "taco_workspace_bytes", "taco_compress", "taco_compress_shards", "taco_compress_shards_fwht",
    "taco_compress_shards_noalloc", "taco_compress_shards_mma",
    "taco_compress_shards_int8", "taco_decompress_reduce_int8",
    "taco_decompress_reduce_mma", "taco_decompress_reduce_mma_ptrs",
    "taco_reduce_recompress_int8_ptrs", "taco_decompress_shards_int8_ptrs",
    "taco_reduce_recompress_batched_ptrs",
    "taco_decompress_reduce", "taco_decompress_reduce_ptrs",
    "taco_reduce_recompress", "taco_reduce_recompress_ptrs",
    "taco_decompress_shards", "taco_decompress_shards_ptrs",
    "taco_e4m3_encode_f32", "taco_e4m3_decode_f32",
    "taco_get_fault", "taco_selftest_wait_timeout",
    "taco_status_string", "taco_abi_version",
)


class TacoError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} "
                         f"({_lib().taco_status_string(status).decode()})")


_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not LIB_PATH.exists():
            raise RuntimeError(
                f"libtaco is not built ({LIB_PATH} missing): run "
                "`python -m grads_taco_compress_gb300.build_lib` first")
        lib = ctypes.CDLL(str(LIB_PATH))
        i64, i32, sz, vp, f32 = (ctypes.c_int64, ctypes.c_int, ctypes.c_size_t,
                                 ctypes.c_void_p, ctypes.c_float)
        sig = {
            "taco_shard_bytes": (sz, [i64, i64, i32]),
            "taco_shard_scales_offset": (sz, [i64, i64, i32]),
            "taco_workspace_bytes": (sz, [i32]),
            "taco_compress": (i32, [vp, i64, i64, i32, f32, i32, vp, vp, vp, sz, vp]),
            "taco_compress_shards": (i32, [vp, i32, i64, i64, i32, f32, i32, vp, vp, vp, sz, vp]),
            "taco_compress_shards_fwht": (i32, [vp, i32, i64, i64, i32, f32, i32, vp, vp, vp, sz, vp]),
            "taco_compress_shards_noalloc": (i32, [vp, i32, i64, i64, i32, f32, i32, vp, vp, vp]),
            "taco_compress_shards_mma": (i32, [vp, i32, i64, i64, i32, f32, i32, vp, vp, vp, sz, vp]),
            "taco_compress_shards_int8": (i32, [vp, i32, i64, i64, i32, f32, i32, vp, vp, vp, sz, vp]),
            "taco_decompress_reduce_int8": (i32, [vp, i32, i64, i64, i32, vp, vp]),
            "taco_decompress_reduce_mma": (i32, [vp, i32, i64, i64, i32, vp, vp]),
            "taco_decompress_reduce_mma_ptrs": (i32, [ctypes.POINTER(vp), i32, i64, i64, i32, vp, vp]),
            "taco_reduce_recompress_int8_ptrs": (i32, [ctypes.POINTER(vp), i32, i64, i64, i32, f32, i32,
                                                       vp, vp, vp, vp, sz, vp]),
            "taco_decompress_shards_int8_ptrs": (i32, [ctypes.POINTER(vp), i32, i64, i64, i32, vp, vp]),
            "taco_reduce_recompress_batched_ptrs": (i32, [ctypes.POINTER(vp), i32, i32, i64, i64, i32, f32,
                                                          i32, i32, vp, vp, vp, sz, vp]),
            "taco_decompress_reduce": (i32, [vp, i32, i64, i64, i32, vp, vp]),
            "taco_decompress_reduce_ptrs": (i32, [ctypes.POINTER(vp), i32, i64, i64, i32, vp, vp]),
            "taco_decompress_shards": (i32, [vp, i32, i64, i64, i32, vp, vp]),
            "taco_decompress_shards_ptrs": (i32, [ctypes.POINTER(vp), i32, i64, i64, i32, vp, vp]),
            "taco_reduce_recompress": (i32, [vp, i32, i64, i64, i32, f32, i32, vp, vp, vp, vp, sz, vp]),
            "taco_reduce_recompress_ptrs": (i32, [ctypes.POINTER(vp), i32, i64, i64, i32, f32, i32,
                                                  vp, vp, vp, vp, sz, vp]),
            "taco_e4m3_encode_f32": (i32, [vp, vp, i64, vp]),
            "taco_e4m3_decode_f32": (i32, [vp, vp, i64, vp]),
            "taco_get_fault": (i32, [ctypes.POINTER(ctypes.c_uint32), i32]),
            "taco_selftest_wait_timeout": (i32, [ctypes.c_uint64, vp, vp]),
            "taco_status_string": (ctypes.c_char_p, [i32]),
            "taco_abi_version": (i32, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def library() -> ctypes.CDLL:
    """The loaded libtaco (raises if it has not been built)."""
    return _lib()


def _check(status: int, what: str) -> None:
    if status != TACO_OK:
        raise TacoError(status, what)


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


# ---------------------------------------------------------------- layout ----
def shard_bytes(N: int, h: int, block: int) -> int:
    return int(_lib().taco_shard_bytes(N, h, block))


def shard_scales_offset(N: int, h: int, block: int) -> int:
    """Byte offset of the (alpha, s) pairs inside a shard."""
    return int(_lib().taco_shard_scales_offset(N, h, block))


def workspace_bytes(P: int) -> int:
    return int(_lib().taco_workspace_bytes(P))


def new_workspace(P: int = MAX_SHARDS, device=None) -> torch.Tensor:
    """A zero-filled workspace for compress calls of up to P shards."""
    return torch.zeros(workspace_bytes(P), dtype=torch.uint8, device=device or "cuda")


def shard_views(bundle: torch.Tensor, P: int, N: int, h: int, block: int):
    """Views (codes u8 [P,N,h], alpha f32 [P,N,K], s f32 [P,N,K]) into a bundle."""
    sb = shard_bytes(N, h, block)
    off = shard_scales_offset(N, h, block)
    K = h // block
    flat = bundle.view(torch.uint8).reshape(-1)[: P * sb].view(P, sb)
    codes = flat[:, : N * h].reshape(P, N, h)
    scales = flat[:, off: off + 8 * N * K].view(torch.float32).view(P, N, K, 2)
    return codes, scales[..., 0], scales[..., 1]


def parse_headers(headers: torch.Tensor) -> np.ndarray:
    """Device or host header bytes [P, 40] -> numpy records."""
    raw = headers.detach().to("cpu").contiguous().view(torch.uint8).numpy().reshape(-1)
    return raw.view(HEADER_DTYPE)


# -------------------------------------------------------------- operator ----
def _compress_shards(entry: str, x: torch.Tensor, block: int, target_energy, variant, bundle,
                     headers, workspace, stream):
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 3 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 CUDA tensor [P, N, h]")
    P, N, h = x.shape
    sb = shard_bytes(N, h, block)
    if bundle is None:
        bundle = torch.empty((P, max(sb, 1)), dtype=torch.uint8, device=x.device)
    if headers is None:
        headers = torch.empty((P, HEADER_BYTES), dtype=torch.uint8, device=x.device)
    if workspace is None:
        workspace = new_workspace(P, x.device)
    st = getattr(_lib(), entry)(_ptr(x), P, N, h, block, float(target_energy), variant,
                                _ptr(bundle), _ptr(headers), _ptr(workspace),
                                workspace.numel(), _stream_ptr(stream))
    _check(st, entry)
    return bundle, headers


def taco_compress_shards(x: torch.Tensor, block: int, target_energy: float = DEFAULT_TARGET_ENERGY,
                         variant: int = VARIANT_DUAL, bundle: torch.Tensor | None = None,
                         headers: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         stream=None):
    """Compress bf16 x [P, N, h] (cuda, contiguous) into a bundle of P shards
    (the tensor-core kernel; the CUDA-core FWHT beyond 2^31 - 256 blocks per
    shard).

    Returns (bundle u8 [P, shard_bytes], headers u8 [P, 40]).
    """
    return _compress_shards("taco_compress_shards", x, block, target_energy, variant, bundle,
                            headers, workspace, stream)


def taco_compress_shards_fwht(x: torch.Tensor, block: int, target_energy: float = DEFAULT_TARGET_ENERGY,
                              variant: int = VARIANT_DUAL, bundle: torch.Tensor | None = None,
                              headers: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                              stream=None):
    """taco_compress_shards with the whole rotation as a CUDA-core FWHT."""
    return _compress_shards("taco_compress_shards_fwht", x, block, target_energy, variant, bundle,
                            headers, workspace, stream)


def taco_compress_shards_mma(x: torch.Tensor, block: int, target_energy: float = DEFAULT_TARGET_ENERGY,
                             variant: int = VARIANT_DUAL, bundle: torch.Tensor | None = None,
                             headers: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                             stream=None):
    """taco_compress_shards with the 64-point Hadamard products on the tensor cores."""
    return _compress_shards("taco_compress_shards_mma", x, block, target_energy, variant, bundle,
                            headers, workspace, stream)


def taco_compress_shards_noalloc(x: torch.Tensor, block: int,
                                 target_energy: float = DEFAULT_TARGET_ENERGY,
                                 variant: int = VARIANT_DUAL, bundle: torch.Tensor | None = None,
                                 headers: torch.Tensor | None = None, stream=None):
    """taco_compress_shards with the library's static scratch instead of a workspace.

    For callers that cannot allocate device memory where they compress; pass
    preallocated ``bundle`` and ``headers`` to allocate nothing at all. At most
    8 shards; calls that overlap on the GPU share the scratch and race.
    """
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 3 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 CUDA tensor [P, N, h]")
    P, N, h = x.shape
    if bundle is None:
        bundle = torch.empty((P, max(shard_bytes(N, h, block), 1)), dtype=torch.uint8, device=x.device)
    if headers is None:
        headers = torch.empty((P, HEADER_BYTES), dtype=torch.uint8, device=x.device)
    st = _lib().taco_compress_shards_noalloc(_ptr(x), P, N, h, block, float(target_energy), variant,
                                             _ptr(bundle), _ptr(headers), _stream_ptr(stream))
    _check(st, "taco_compress_shards_noalloc")
    return bundle, headers


def taco_compress(x: torch.Tensor, block: int, target_energy: float = DEFAULT_TARGET_ENERGY,
                  variant: int = VARIANT_DUAL, shard: torch.Tensor | None = None,
                  header: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None):
    """Compress one bf16 tensor x [N, h]; returns (shard u8 [shard_bytes], header u8 [40])."""
    if x.dim() != 2:
        raise ValueError("x must be [N, h]")
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 CUDA tensor")
    N, h = x.shape
    sb = shard_bytes(N, h, block)
    if shard is None:
        shard = torch.empty(max(sb, 1), dtype=torch.uint8, device=x.device)
    if header is None:
        header = torch.empty(HEADER_BYTES, dtype=torch.uint8, device=x.device)
    if workspace is None:
        workspace = new_workspace(1, x.device)
    st = _lib().taco_compress(_ptr(x), N, h, block, float(target_energy), variant, _ptr(shard),
                              _ptr(header), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(st, "taco_compress")
    return shard, header


def _decompress_reduce(entry: str, bundle: torch.Tensor, P: int, N: int, h: int, block: int,
                       out, stream) -> torch.Tensor:
    if not bundle.is_cuda:
        raise ValueError("bundle must be a CUDA tensor")
    if out is None:
        out = torch.empty((N, h), dtype=torch.bfloat16, device=bundle.device)
    st = getattr(_lib(), entry)(_ptr(bundle), P, N, h, block, _ptr(out), _stream_ptr(stream))
    _check(st, entry)
    return out


def taco_decompress_reduce(bundle: torch.Tensor, P: int, N: int, h: int, block: int,
                           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Sum of the P reconstructions of a bundle as bf16 [N, h]."""
    return _decompress_reduce("taco_decompress_reduce", bundle, P, N, h, block, out, stream)


def taco_compress_shards_int8(x: torch.Tensor, block: int, target_energy: float = DEFAULT_TARGET_ENERGY,
                              variant: int = VARIANT_DUAL, bundle: torch.Tensor | None = None,
                              headers: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                              stream=None):
    """taco_compress_shards_mma with INT8 fallback codes (Q_max 127)."""
    return _compress_shards("taco_compress_shards_int8", x, block, target_energy, variant, bundle,
                            headers, workspace, stream)


def taco_decompress_reduce_mma(bundle: torch.Tensor, P: int, N: int, h: int, block: int,
                               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """taco_decompress_reduce with the inverse rotation on the tensor cores (block 64, 128)."""
    return _decompress_reduce("taco_decompress_reduce_mma", bundle, P, N, h, block, out, stream)


def taco_decompress_reduce_mma_ptrs(shards, N: int, h: int, block: int,
                                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """taco_decompress_reduce_mma with P separate shard tensors."""
    P = len(shards)
    if out is None:
        out = torch.empty((N, h), dtype=torch.bfloat16, device=shards[0].device)
    arr = (ctypes.c_void_p * max(P, 1))(*[_ptr(s) for s in shards])
    st = _lib().taco_decompress_reduce_mma_ptrs(arr, P, N, h, block, _ptr(out), _stream_ptr(stream))
    _check(st, "taco_decompress_reduce_mma_ptrs")
    return out


def taco_decompress_reduce_int8(bundle: torch.Tensor, P: int, N: int, h: int, block: int,
                                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """taco_decompress_reduce of a bundle with INT8 fallback codes."""
    return _decompress_reduce("taco_decompress_reduce_int8", bundle, P, N, h, block, out, stream)


def taco_decompress_reduce_ptrs(shards, N: int, h: int, block: int,
                                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """As taco_decompress_reduce with P separate shard tensors."""
    P = len(shards)
    if out is None:
        out = torch.empty((N, h), dtype=torch.bfloat16, device=shards[0].device)
    arr = (ctypes.c_void_p * max(P, 1))(*[_ptr(s) for s in shards])
    st = _lib().taco_decompress_reduce_ptrs(arr, P, N, h, block, _ptr(out), _stream_ptr(stream))
    _check(st, "taco_decompress_reduce_ptrs")
    return out


def taco_decompress_shards(bundle: torch.Tensor, P: int, N: int, h: int, block: int,
                           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Each of the P shards of a bundle reconstructed on its own: bf16 [P, N, h]."""
    if not bundle.is_cuda:
        raise ValueError("bundle must be a CUDA tensor")
    if out is None:
        out = torch.empty((P, N, h), dtype=torch.bfloat16, device=bundle.device)
    st = _lib().taco_decompress_shards(_ptr(bundle), P, N, h, block, _ptr(out), _stream_ptr(stream))
    _check(st, "taco_decompress_shards")
    return out


def taco_decompress_shards_ptrs(shards, N: int, h: int, block: int,
                                out: torch.Tensor | None = None, stream=None,
                                entry: str = "taco_decompress_shards_ptrs") -> torch.Tensor:
    """As taco_decompress_shards with P separate shard tensors."""
    P = len(shards)
    if out is None:
        out = torch.empty((P, N, h), dtype=torch.bfloat16, device=shards[0].device)
    arr = (ctypes.c_void_p * max(P, 1))(*[_ptr(s) for s in shards])
    st = getattr(_lib(), entry)(arr, P, N, h, block, _ptr(out), _stream_ptr(stream))
    _check(st, entry)
    return out


def taco_decompress_shards_int8_ptrs(shards, N: int, h: int, block: int,
                                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """taco_decompress_shards_ptrs for shards with INT8 fallback codes."""
    return taco_decompress_shards_ptrs(shards, N, h, block, out, stream,
                                       entry="taco_decompress_shards_int8_ptrs")


def taco_reduce_recompress(bundle: torch.Tensor, P: int, N: int, h: int, block: int,
                           target_energy: float = DEFAULT_TARGET_ENERGY, variant: int = VARIANT_DUAL,
                           shard: torch.Tensor | None = None, header: torch.Tensor | None = None,
                           out: torch.Tensor | None = None, want_bf16: bool = False,
                           workspace: torch.Tensor | None = None, stream=None):
    """Sum the P shards of a bundle and compress the sum into one shard.

    Returns (shard u8, header u8 [40], bf16 sum or None).
    """
    if not bundle.is_cuda:
        raise ValueError("bundle must be a CUDA tensor")
    dev = bundle.device
    if shard is None:
        shard = torch.empty(max(shard_bytes(N, h, block), 1), dtype=torch.uint8, device=dev)
    if header is None:
        header = torch.empty(HEADER_BYTES, dtype=torch.uint8, device=dev)
    if out is None and want_bf16:
        out = torch.empty((N, h), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = new_workspace(1, dev)
    st = _lib().taco_reduce_recompress(_ptr(bundle), P, N, h, block, float(target_energy), variant,
                                       _ptr(shard), _ptr(header), _ptr(out), _ptr(workspace),
                                       workspace.numel(), _stream_ptr(stream))
    _check(st, "taco_reduce_recompress")
    return shard, header, out


def taco_reduce_recompress_ptrs(shards, N: int, h: int, block: int,
                                target_energy: float = DEFAULT_TARGET_ENERGY,
                                variant: int = VARIANT_DUAL, shard: torch.Tensor | None = None,
                                header: torch.Tensor | None = None, out: torch.Tensor | None = None,
                                workspace: torch.Tensor | None = None, stream=None,
                                entry: str = "taco_reduce_recompress_ptrs"):
    """As taco_reduce_recompress with P separate shard tensors."""
    P = len(shards)
    dev = shards[0].device
    if shard is None:
        shard = torch.empty(max(shard_bytes(N, h, block), 1), dtype=torch.uint8, device=dev)
    if header is None:
        header = torch.empty(HEADER_BYTES, dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = new_workspace(1, dev)
    arr = (ctypes.c_void_p * max(P, 1))(*[_ptr(s) for s in shards])
    st = getattr(_lib(), entry)(arr, P, N, h, block, float(target_energy), variant,
                                _ptr(shard), _ptr(header), _ptr(out), _ptr(workspace),
                                workspace.numel(), _stream_ptr(stream))
    _check(st, entry)
    return shard, header, out


def taco_reduce_recompress_batched_ptrs(shards, Y: int, N: int, h: int, block: int,
                                        target_energy: float = DEFAULT_TARGET_ENERGY,
                                        variant: int = VARIANT_DUAL, code_format: int = FORMAT_E4M3,
                                        shards_out: torch.Tensor | None = None,
                                        headers: torch.Tensor | None = None,
                                        workspace: torch.Tensor | None = None, stream=None):
    """Y reduce-recompress operations in one launch; shards holds Y*P tensors,
    reduction y takes shards[y*P:(y+1)*P]. Returns (shards_out u8 [Y, shard_bytes],
    headers u8 [Y, 40])."""
    if len(shards) % Y:
        raise ValueError("len(shards) must be a multiple of Y")
    P = len(shards) // Y
    dev = shards[0].device
    if shards_out is None:
        shards_out = torch.empty((Y, max(shard_bytes(N, h, block), 1)), dtype=torch.uint8, device=dev)
    if headers is None:
        headers = torch.empty((Y, HEADER_BYTES), dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = new_workspace(Y, dev)
    arr = (ctypes.c_void_p * max(len(shards), 1))(*[_ptr(s) for s in shards])
    st = _lib().taco_reduce_recompress_batched_ptrs(arr, Y, P, N, h, block, float(target_energy), variant,
                                                     code_format, _ptr(shards_out), _ptr(headers),
                                                     _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(st, "taco_reduce_recompress_batched_ptrs")
    return shards_out, headers


def taco_reduce_recompress_int8_ptrs(shards, N: int, h: int, block: int,
                                     target_energy: float = DEFAULT_TARGET_ENERGY,
                                     variant: int = VARIANT_DUAL, shard: torch.Tensor | None = None,
                                     header: torch.Tensor | None = None, out: torch.Tensor | None = None,
                                     workspace: torch.Tensor | None = None, stream=None):
    """taco_reduce_recompress_ptrs with INT8 fallback codes in and out."""
    return taco_reduce_recompress_ptrs(shards, N, h, block, target_energy, variant, shard, header,
                                       out, workspace, stream, entry="taco_reduce_recompress_int8_ptrs")


def taco_e4m3_encode_f32(x: torch.Tensor, stream=None) -> torch.Tensor:
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 CUDA tensor")
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(_lib().taco_e4m3_encode_f32(_ptr(x), _ptr(out), x.numel(), _stream_ptr(stream)),
           "taco_e4m3_encode_f32")
    return out


def taco_e4m3_decode_f32(codes: torch.Tensor, stream=None) -> torch.Tensor:
    if codes.dtype != torch.uint8 or not codes.is_cuda or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 CUDA tensor")
    out = torch.empty(codes.shape, dtype=torch.float32, device=codes.device)
    _check(_lib().taco_e4m3_decode_f32(_ptr(codes), _ptr(out), codes.numel(), _stream_ptr(stream)),
           "taco_e4m3_decode_f32")
    return out


def taco_get_fault(clear: bool = False) -> int:
    """Device fault bits of the current device (synchronises with it)."""
    bits = ctypes.c_uint32(0)
    _check(_lib().taco_get_fault(ctypes.byref(bits), int(clear)), "taco_get_fault")
    return int(bits.value)


def taco_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Run the bounded-wait self-test; returns the status word (1 = timed out)."""
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    _check(_lib().taco_selftest_wait_timeout(int(limit_ns), _ptr(status), _stream_ptr(stream)),
           "taco_selftest_wait_timeout")
    return int(status.item())

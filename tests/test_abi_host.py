"""The C ABI without a GPU: exports, layout, and host-side argument checks.

Every call below is rejected by the host checks before any CUDA call, so the
fake addresses are never dereferenced; no case here reaches a launch.
"""

from __future__ import annotations

import ctypes
import pathlib
import re

import pytest
import torch

from grads_taco_compress_gb300 import binding as tb

# Fake addresses are only safe where no kernel could ever be launched.
no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                                 reason="fake-address host checks run on machines without a GPU")

ROOT = pathlib.Path(__file__).resolve().parent.parent
OK, NULL, SHAPE, BLOCK, ALIGN, ARG, CUDA, WS = range(8)
A = 0x10000          # a 256-byte aligned fake device address
WSB = 16 * 16400     # larger than any workspace the library asks for


@pytest.fixture(scope="module")
def lib():
    if not tb.LIB_PATH.exists():
        from grads_taco_compress_gb300 import build_lib
        build_lib.build()
    return tb.library()


def _declared_functions():
    text = (ROOT / "include" / "taco.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(taco_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert sorted(tb.EXPORTED_SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.taco_abi_version() == 1


def test_shard_layout(lib):
    def pad(v):
        return (v + 255) // 256 * 256
    for N, h, n in [(512, 1024, 128), (8192, 1600, 64), (16384, 3584, 128), (1, 64, 64), (3, 768, 256),
                    (0, 256, 128)]:
        K = h // n
        off = pad(N * h)
        assert lib.taco_shard_scales_offset(N, h, n) == off
        assert lib.taco_shard_bytes(N, h, n) == off + pad(8 * N * K)
    for N, h, n in [(4, 100, 64), (4, 128, 100), (-1, 128, 64), (4, 0, 64)]:
        assert lib.taco_shard_bytes(N, h, n) == 0
    assert lib.taco_workspace_bytes(0) == 0 and lib.taco_workspace_bytes(17) == 0
    assert lib.taco_workspace_bytes(1) == 16 and lib.taco_workspace_bytes(16) == 256 <= WSB


def _compress(lib, x=A, P=1, N=4, h=256, block=128, E=4096.0, variant=0, bundle=A * 64,
              headers=A * 128, ws=A * 256, wsb=WSB, entry="taco_compress_shards"):
    return getattr(lib, entry)(x, P, N, h, block, E, variant, bundle, headers, ws, wsb, None)


@no_gpu_only
@pytest.mark.parametrize("kwargs,status", [
    (dict(block=100), BLOCK), (dict(block=32), BLOCK), (dict(block=512), BLOCK),
    (dict(h=130, block=64), SHAPE), (dict(N=-1), SHAPE), (dict(h=0), SHAPE),
    (dict(N=1 << 34, h=1 << 10), SHAPE),
    (dict(P=0), ARG), (dict(P=17), ARG), (dict(variant=3), ARG), (dict(variant=-1), ARG),
    (dict(E=0.0), ARG), (dict(E=-1.0), ARG), (dict(E=float("nan")), ARG),
    (dict(E=float("inf")), ARG), (dict(E=2.0 ** 121), ARG),
    (dict(headers=None), NULL), (dict(ws=None), WS), (dict(wsb=15), WS),
    (dict(x=None), NULL), (dict(bundle=None), NULL),
    (dict(x=A + 8), ALIGN), (dict(bundle=A * 64 + 4), ALIGN), (dict(headers=A * 128 + 4), ALIGN),
    (dict(ws=A * 256 + 8), ALIGN),
    (dict(x=A, bundle=A + 64), ARG),                  # input and output overlap
])
@pytest.mark.parametrize("entry", ["taco_compress_shards", "taco_compress_shards_fwht"])
def test_compress_rejects(lib, kwargs, status, entry):
    assert status not in (OK, CUDA)
    assert _compress(lib, entry=entry, **kwargs) == status


@no_gpu_only
@pytest.mark.parametrize("kwargs,status", [
    (dict(block=100), BLOCK), (dict(h=130, block=64), SHAPE), (dict(N=-1), SHAPE),
    (dict(P=0), ARG), (dict(variant=3), ARG), (dict(E=float("nan")), ARG),
    (dict(N=1 << 26, h=1 << 12, block=64, bundle=1 << 44), SHAPE),   # 2^32 blocks: beyond 32-bit TMA rows
    (dict(headers=None), NULL), (dict(ws=None), WS), (dict(x=A + 8), ALIGN),
    (dict(x=A, bundle=A + 64), ARG),
])
def test_compress_mma_rejects(lib, kwargs, status):
    args = dict(x=A, P=1, N=4, h=256, block=128, E=4096.0, variant=0, bundle=A * 64,
                headers=A * 128, ws=A * 256, wsb=WSB)
    args.update(kwargs)
    st = lib.taco_compress_shards_mma(args["x"], args["P"], args["N"], args["h"], args["block"],
                                      args["E"], args["variant"], args["bundle"], args["headers"],
                                      args["ws"], args["wsb"], None)
    assert st == status


@no_gpu_only
def test_decompress_mma_rejects(lib):
    assert lib.taco_decompress_reduce_mma(A, 2, 4, 256, 256, A * 1024, None) == BLOCK
    assert lib.taco_decompress_reduce_mma(A, 2, 4, 200, 64, A * 1024, None) == SHAPE
    assert lib.taco_decompress_reduce_mma(A, 17, 4, 256, 128, A * 1024, None) == ARG
    assert lib.taco_decompress_reduce_mma(None, 2, 4, 256, 128, A * 1024, None) == NULL
    assert lib.taco_decompress_reduce_mma(A, 2, 4, 256, 128, A * 1024 + 2, None) == ALIGN
    assert lib.taco_decompress_reduce_mma(A, 2, 4, 256, 128, A + 512, None) == ARG
    assert lib.taco_decompress_reduce_int8(A, 2, 4, 256, 128, A * 1024 + 2, None) == ALIGN
    assert lib.taco_compress_shards_int8(A, 1, 4, 256, 128, 4096.0, 3, A * 64, A * 128, A * 256,
                                         WSB, None) == ARG


@no_gpu_only
def test_single_compress_rejects(lib):
    assert lib.taco_compress(A, 4, 256, 100, 4096.0, 0, A * 64, A * 128, A * 256, WSB, None) == BLOCK
    assert lib.taco_compress(A + 2, 4, 256, 128, 4096.0, 0, A * 64, A * 128, A * 256, WSB, None) == ALIGN


def _decompress(lib, bundle=A, P=2, N=4, h=256, block=128, out=A * 1024):
    return lib.taco_decompress_reduce(bundle, P, N, h, block, out, None)


@no_gpu_only
@pytest.mark.parametrize("kwargs,status", [
    (dict(block=96), BLOCK), (dict(h=200, block=64), SHAPE), (dict(N=-3), SHAPE),
    (dict(P=0), ARG), (dict(P=17), ARG), (dict(bundle=None), NULL), (dict(out=None), NULL),
    (dict(out=A * 1024 + 2), ALIGN), (dict(bundle=A + 8), ALIGN),
    (dict(bundle=A, out=A + 512), ARG),               # output inside the bundle
])
def test_decompress_rejects(lib, kwargs, status):
    assert _decompress(lib, **kwargs) == status


@no_gpu_only
def test_decompress_empty_is_ok_without_launch(lib):
    # N == 0 returns before any device work, even with no buffers at all
    assert _decompress(lib, bundle=None, N=0, out=None) == OK


@no_gpu_only
def test_decompress_ptrs_rejects(lib):
    arr = (ctypes.c_void_p * 3)(A, A * 64, None)
    assert lib.taco_decompress_reduce_ptrs(arr, 3, 4, 256, 128, A * 1024, None) == NULL
    arr = (ctypes.c_void_p * 2)(A, A * 64 + 8)
    assert lib.taco_decompress_reduce_ptrs(arr, 2, 4, 256, 128, A * 1024, None) == ALIGN
    assert lib.taco_decompress_reduce_ptrs(None, 2, 4, 256, 128, A * 1024, None) == NULL
    arr = (ctypes.c_void_p * 2)(A, A * 64)
    assert lib.taco_decompress_reduce_ptrs(arr, 0, 4, 256, 128, A * 1024, None) == ARG


@no_gpu_only
def test_codec_rejects(lib):
    assert lib.taco_e4m3_encode_f32(A, A * 8, -1, None) == SHAPE
    assert lib.taco_e4m3_encode_f32(None, A * 8, 10, None) == NULL
    assert lib.taco_e4m3_encode_f32(A + 2, A * 8, 10, None) == ALIGN
    assert lib.taco_e4m3_decode_f32(A, None, 10, None) == NULL
    assert lib.taco_e4m3_decode_f32(A, A * 8 + 1, 10, None) == ALIGN
    assert lib.taco_e4m3_encode_f32(None, None, 0, None) == OK


def test_status_strings(lib):
    for s in range(8):
        assert lib.taco_status_string(s)
    assert b"unknown" in lib.taco_status_string(99)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(tb, "LIB_PATH", tmp_path / "missing.so")
    monkeypatch.setattr(tb, "_LIB", None)
    with pytest.raises(RuntimeError, match="not built"):
        tb.shard_bytes(4, 256, 128)


@no_gpu_only
def test_fault_api_rejects(lib):
    assert lib.taco_get_fault(None, 0) == NULL
    assert lib.taco_selftest_wait_timeout(1000, None, None) == NULL
    assert lib.taco_selftest_wait_timeout(1000, A + 2, None) == ALIGN
    assert lib.taco_selftest_wait_timeout(0, A, None) == ARG
    assert lib.taco_selftest_wait_timeout(3_000_000_000, A, None) == ARG


@no_gpu_only
def test_reduce_recompress_rejects(lib):
    def call(bundle=A, P=2, N=4, h=256, block=128, E=4096.0, variant=0, shard=A * 64, hdr=A * 128,
             out=None, ws=A * 256, wsb=WSB):
        return lib.taco_reduce_recompress(bundle, P, N, h, block, E, variant, shard, hdr, out, ws, wsb, None)
    assert call(block=100) == BLOCK
    assert call(h=200, block=64) == SHAPE
    assert call(P=0) == ARG and call(P=17) == ARG
    assert call(variant=3) == ARG and call(E=0.0) == ARG and call(E=float("nan")) == ARG
    assert call(E=2.0 ** 121) == ARG
    assert call(hdr=None) == NULL and call(ws=None) == WS and call(wsb=15) == WS
    assert call(bundle=None) == NULL and call(shard=None) == NULL
    assert call(shard=A * 64 + 8) == ALIGN and call(out=A * 512 + 4) == ALIGN
    assert call(shard=A + 256) == ARG                     # output shard inside the inputs
    assert call(out=A * 64) == ARG                        # bf16 output over the output shard
    arr = (ctypes.c_void_p * 2)(A, None)
    assert lib.taco_reduce_recompress_ptrs(arr, 2, 4, 256, 128, 4096.0, 0, A * 64, A * 128, None,
                                           A * 256, WSB, None) == NULL

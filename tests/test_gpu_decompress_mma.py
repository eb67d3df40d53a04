"""Tensor-core decompress-reduce (taco_decompress_reduce_mma) against the oracle.

Bar: reconstruction within 1e-3 relative RMS of the oracle (the contract of
taco_decompress_reduce), and the same against the CUDA-core kernel; sizes
leave a ragged last tile of 128 blocks and P covers one and several shard
groups (4 shards per group at n = 64, 2 at n = 128).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O
from test_gpu_parity import E_STAR, bundle_from_arrays, host_bits

pytestmark = pytest.mark.gpu

MMA = tb.taco_decompress_reduce_mma


def _check(codes, alpha, s, block):
    P, N, h = codes.shape
    bundle = bundle_from_arrays(codes, alpha, s, block)
    got = O.bf16_bits_to_f64(host_bits(MMA(bundle, P, N, h, block)))
    want = O.bf16_bits_to_f64(O.decompress_reduce(codes, alpha, s, block))
    parity.compare_recon(got, want)
    ref = O.bf16_bits_to_f64(host_bits(tb.taco_decompress_reduce(bundle, P, N, h, block)))
    parity.compare_recon(got, ref, "against the CUDA-core kernel")
    assert np.mean(got == ref) > 0.99
    return got


def test_mma_decompress_one_tile():
    codes, alpha, s = W.make_random_bundle(128, 64, 64, 1, seed=50)
    _check(codes, alpha, s, 64)


@pytest.mark.parametrize("block,P", [(64, 1), (64, 3), (64, 4), (64, 5), (64, 9), (64, 16),
                                     (128, 1), (128, 2), (128, 3), (128, 8), (128, 16)])
def test_mma_decompress_random_bundles(block, P):
    N, h = 27, 5 * block                     # 135 blocks: one full tile and a ragged one
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=block + P)
    _check(codes, alpha, s, block)


@pytest.mark.parametrize("name,rows", [("tiny-512x1024", 96), ("gpt2-1.5b-act", 37),
                                       ("gpt3-6.7b-act", 29), ("qwen-7b-long", 19)])
def test_mma_decompress_from_oracle_codes(name, rows):
    w = W.WORKLOADS[name]
    x = W.make_shards(w, N=rows)
    parts = [O.compress(x[p], w.block, E_STAR) for p in range(w.P)]
    codes = np.stack([c for c, _, _, _ in parts])
    alpha = np.stack([a for _, a, _, _ in parts])
    s = np.stack([sc for _, _, sc, _ in parts])
    _check(codes, alpha, s, w.block)


def test_mma_decompress_every_code():
    """All 254 finite codes in one block row, one shard, unit scales."""
    block = 128
    codes = np.concatenate([np.arange(0, 127), np.arange(128, 255)]).astype(np.uint8)
    codes = np.concatenate([codes, np.zeros(2 * block - codes.size, np.uint8)]).reshape(1, 1, 2 * block)
    alpha = np.ones((1, 1, 2), np.float32)
    s = np.ones((1, 1, 2), np.float32)
    _check(codes, alpha, s, block)


def test_mma_decompress_ptrs_equals_bundle():
    block, P, N, h = 64, 6, 45, 640
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=7)
    bundle = bundle_from_arrays(codes, alpha, s, block)
    a = MMA(bundle, P, N, h, block)
    b = tb.taco_decompress_reduce_mma_ptrs([bundle[p].clone() for p in range(P)], N, h, block)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_mma_decompress_guards_empty_and_block_256():
    block, P, N, h = 128, 3, 19, 384
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=8)
    bundle = bundle_from_arrays(codes, alpha, s, block)
    guard = 4096
    big = torch.full((N * h + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
    MMA(bundle, P, N, h, block, out=big[guard: guard + N * h].view(N, h))
    torch.cuda.synchronize()
    assert bool((big[:guard] == -7.0).all()) and bool((big[-guard:] == -7.0).all())
    MMA(bundle, P, 0, h, block, out=big[guard: guard + 16].view(1, 16)[:0])   # N = 0: nothing
    with pytest.raises(tb.TacoError):
        MMA(bundle, 1, 1, 256, 256)


@pytest.mark.parametrize("name", ["tiny-512x1024", "gpt2-1.5b-act", "gpt3-6.7b-act", "qwen-7b-long"])
def test_mma_decompress_full_size_every_element(name, oracle_rows):
    """The benchmark's launch shape at full size: every element against the
    oracle and against the CUDA-core kernel."""
    w = W.WORKLOADS[name]
    codes, alpha, s = W.make_random_bundle(w.N, w.h, w.block, w.P, seed=9)
    bundle = bundle_from_arrays(codes, alpha, s, w.block)
    got = host_bits(MMA(bundle, w.P, w.N, w.h, w.block))
    want = oracle_rows.decompress_reduce(codes, alpha, s, w.block)
    parity.compare_recon(O.bf16_bits_to_f64(got), O.bf16_bits_to_f64(want))
    ref = host_bits(tb.taco_decompress_reduce(bundle, w.P, w.N, w.h, w.block))
    parity.compare_recon(O.bf16_bits_to_f64(got), O.bf16_bits_to_f64(ref), "against the CUDA-core kernel")
    assert np.all(np.isfinite(O.bf16_bits_to_f64(got)))


def test_mma_decompress_no_wait_timed_out():
    assert tb.taco_get_fault() & 16 == 0

"""taco_reduce_recompress against the oracle's reduce_recompress.

The fused kernel sums P shards in the rotated domain and compresses the sum
again without an inverse and forward transform; the oracle reconstructs the
sum in fp64 and runs the compress steps on it (the plain composition)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O
from test_gpu_parity import bundle_from_arrays, gpu_compress, host_bits

pytestmark = pytest.mark.gpu
E_STAR = 4096.0


def gpu_recompress(codes, alpha, s, block, variant=tb.VARIANT_DUAL, target=E_STAR, want_bf16=False):
    P, N, h = codes.shape
    bundle = bundle_from_arrays(codes, alpha, s, block)
    shard, header, out = tb.taco_reduce_recompress(bundle, P, N, h, block, target, variant,
                                                   want_bf16=want_bf16)
    rc, ra, rs = tb.shard_views(shard.view(1, -1), 1, N, h, block)
    torch.cuda.synchronize()
    return (rc[0].cpu().numpy(), ra[0].cpu().numpy(), rs[0].cpu().numpy(),
            tb.parse_headers(header)[0], out, bundle)


def check(codes, alpha, s, block, variant=tb.VARIANT_DUAL, target=E_STAR):
    rc, ra, rs, hdr, _, _ = gpu_recompress(codes, alpha, s, block, variant, target)
    oc, oa, os_, oh = O.reduce_recompress(codes, alpha, s, block, target, variant)
    parity.compare_codes(rc, oc, "recompressed codes")
    parity.compare_scales(ra, oa, "recompressed alpha")
    parity.compare_scales(rs, os_, "recompressed s")
    assert hdr["N"] == codes.shape[1] and hdr["h"] == codes.shape[2] and hdr["block"] == block
    assert abs(hdr["s_max"] - oh["s_max"]) <= 1e-6 * max(oh["s_max"], 1.0)
    near_one = np.count_nonzero(np.abs(os_.astype(np.float64) - 1.0) < 1e-6)
    assert abs(int(hdr["n_clamped"]) - oh["n_clamped"]) <= near_one


def oracle_bundle(x, block):
    parts = [O.compress(x[p], block, E_STAR) for p in range(x.shape[0])]
    return (np.stack([c for c, _, _, _ in parts]), np.stack([a for _, a, _, _ in parts]),
            np.stack([sc for _, _, sc, _ in parts]))


@pytest.mark.parametrize("name,rows", [("tiny-512x1024", 64), ("gpt2-1.5b-act", 37), ("gpt3-6.7b-act", 29),
                                       ("gpt3-6.7b-grad", 23), ("qwen-7b-long", 19)])
def test_recompress_small(name, rows):
    w = W.WORKLOADS[name]
    x = W.make_shards(w, N=rows)
    check(*oracle_bundle(x, w.block), w.block)


@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX, tb.VARIANT_STATIC])
def test_recompress_random_bundles(block, variant):
    codes, alpha, s = W.make_random_bundle(21, 3 * block, block, 5, seed=block + variant)
    for target in (E_STAR, 2.0):
        check(codes, alpha, s, block, variant, target)


def test_recompress_bf16_side_output_equals_decompress_reduce():
    block, P, N, h = 128, 4, 45, 768
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=9)
    _, _, _, _, out, bundle = gpu_recompress(codes, alpha, s, block, want_bf16=True)
    ref = tb.taco_decompress_reduce(bundle, P, N, h, block)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), host_bits(ref))


@pytest.mark.parametrize("block", [64, 128, 256])
def test_recompress_of_spike_blocks_is_exact(block):
    rng = np.random.default_rng(block)
    xv = np.zeros((1, 6, 2 * block), dtype=np.float32)
    for r in range(6):
        xv[0, r, int(rng.integers(2 * block))] = (-1.0) ** r * 0.25 * (r + 1)
    x = W.f32_to_bf16_bits(xv)
    codes, alpha, s, _, _ = gpu_compress(x, block)
    rc, ra, rs, _, _, _ = gpu_recompress(codes, alpha, s, block)
    assert np.array_equal(rc, codes[0])
    assert np.allclose(ra, alpha[0], rtol=3e-7) and np.array_equal(rs, s[0])


def test_recompress_ptrs_equals_bundle():
    block, P, N, h = 64, 3, 33, 640
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=4)
    rc, ra, rs, _, _, bundle = gpu_recompress(codes, alpha, s, block)
    shards = [bundle[p].clone() for p in range(P)]
    shard, header, _ = tb.taco_reduce_recompress_ptrs(shards, N, h, block)
    c2, a2, s2 = tb.shard_views(shard.view(1, -1), 1, N, h, block)
    torch.cuda.synchronize()
    assert np.array_equal(c2[0].cpu().numpy(), rc)
    assert np.array_equal(a2[0].cpu().numpy(), ra) and np.array_equal(s2[0].cpu().numpy(), rs)


@pytest.mark.parametrize("name", ["tiny-512x1024", "gpt2-1.5b-act", "gpt3-6.7b-act", "gpt3-6.7b-grad",
                                  "qwen-7b-long"])
def test_recompress_full_size_every_element(name, oracle_rows):
    """Every code, alpha and s of the full-size reduce-recompress of a
    generated bundle against the oracle (run unchanged over row ranges in
    worker processes), and the header against the GPU's own s."""
    w = W.WORKLOADS[name]
    codes, alpha, s = W.make_random_bundle(w.N, w.h, w.block, w.P, seed=6)
    rc, ra, rs, hdr, _, _ = gpu_recompress(codes, alpha, s, w.block)
    oc, oa, os_ = oracle_rows.reduce_recompress(codes, alpha, s, w.block, E_STAR)
    stats = parity.compare_codes(rc, oc, f"{name} recompressed codes")
    parity.compare_scales(ra, oa, f"{name} alpha")
    parity.compare_scales(rs, os_, f"{name} s")
    assert hdr["s_max"] == rs.max() and hdr["n_clamped"] == np.count_nonzero(rs > 1.0)
    print(f"\nPARITY {name} reduce-recompress: {stats}")


@pytest.mark.parametrize("Y,P,block,fmt", [(4, 4, 64, tb.FORMAT_E4M3), (2, 8, 128, tb.FORMAT_E4M3),
                                           (3, 5, 256, tb.FORMAT_E4M3), (4, 4, 128, tb.FORMAT_INT8),
                                           (1, 16, 64, tb.FORMAT_E4M3)])
def test_batched_recompress_equals_single_calls(Y, P, block, fmt):
    """Y reductions in one launch: each output equals the single-call result."""
    from test_gpu_parity import bundle_from_arrays
    N, h = 23, 3 * block
    shards = []
    for y in range(Y):
        codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=100 * y + block + P)
        if fmt == tb.FORMAT_INT8:
            codes = (codes.astype(np.int64) % 201 - 100).astype(np.int8).view(np.uint8)
        b = bundle_from_arrays(codes, alpha, s, block)
        shards += [b[p] for p in range(P)]
    out, headers = tb.taco_reduce_recompress_batched_ptrs(shards, Y, N, h, block, 900.0, tb.VARIANT_DUAL, fmt)
    single = tb.taco_reduce_recompress_ptrs if fmt == tb.FORMAT_E4M3 else tb.taco_reduce_recompress_int8_ptrs
    off = tb.shard_scales_offset(N, h, block)
    nbytes_scales = N * (h // block) * 8
    for y in range(Y):
        sh, hd, _ = single(shards[y * P:(y + 1) * P], N, h, block, 900.0, tb.VARIANT_DUAL)
        torch.cuda.synchronize()
        # codes and scale pairs (the padding between and after them is never written)
        assert torch.equal(out[y, :N * h], sh[:N * h])
        assert torch.equal(out[y, off:off + nbytes_scales], sh[off:off + nbytes_scales])
        assert torch.equal(headers[y], hd)

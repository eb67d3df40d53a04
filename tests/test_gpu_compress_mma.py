"""Tensor-core compress (taco_compress_shards_mma) against the CPU oracle.

Same parity bar as the CUDA-core compress: codes at least 99.99% equal and
otherwise one E4M3 step apart, alpha and s within 1e-6 relative. The sizes
leave a ragged last tile of 128 blocks and give some CTAs no tile at all;
the full-size cases run many tiles per CTA, so every barrier phase wraps.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O
import test_gpu_parity as GP
from test_gpu_parity import E_STAR, check_compress_against_oracle, dev_bf16, gpu_compress, report

pytestmark = pytest.mark.gpu

MMA = tb.taco_compress_shards_mma


def test_mma_one_tile():
    """128 blocks of 64: exactly one full tile, one CTA."""
    rng = np.random.default_rng(40)
    x = W.f32_to_bf16_bits(rng.normal(0, 0.1, size=(1, 128, 64)).astype(np.float32))
    check_compress_against_oracle(x, 64, entry=MMA)


@pytest.mark.parametrize("block", [64, 128, 256])
def test_mma_less_than_one_tile(block):
    rng = np.random.default_rng(41 + block)
    x = W.f32_to_bf16_bits(rng.laplace(0, 0.05, size=(2, 3, 2 * block)).astype(np.float32))
    check_compress_against_oracle(x, block, entry=MMA)


SMALL = [
    ("tiny-512x1024", 512),
    ("gpt2-1.5b-act", 37),
    ("gpt3-6.7b-act", 29),
    ("gpt3-6.7b-grad", 23),
    ("qwen-7b-long", 19),
]


@pytest.mark.parametrize("name,rows", SMALL)
def test_mma_small(name, rows):
    w = W.WORKLOADS[name]
    x = W.make_shards(w, N=rows, P=min(w.P, 3))
    _, _, _, _, stats = check_compress_against_oracle(x, w.block, entry=MMA)
    assert all(s["equal_fraction"] >= parity.CODE_EQUAL_FRACTION for s in stats)


@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX, tb.VARIANT_STATIC])
def test_mma_variants_and_targets(block, variant):
    rng = np.random.default_rng(block + 10 * variant + 1)
    v = rng.laplace(0, 0.02, size=(2, 41, 3 * block))
    v[:, :, 5] *= 300.0                              # an outlier channel -> clamped blocks
    x = W.f32_to_bf16_bits(v.astype(np.float32))
    for target in (E_STAR, 1.0, 150.0):
        check_compress_against_oracle(x, block, variant, target, entry=MMA)


@pytest.mark.parametrize("block", [64, 128, 256])
def test_mma_closed_form_blocks(block):
    GP.test_compress_closed_form_blocks(block, entry=MMA)


@pytest.mark.parametrize("block", [64, 128, 256])
def test_mma_static_hadamard_rows(block):
    """STATIC: a block equal to a scaled Hadamard row reaches Q_max exactly."""
    H = O.sylvester_hadamard(block).astype(np.float32)
    ks = [0, 1, block // 2, block - 1]
    rows = np.stack([0.25 * H[k] for k in ks] + [-4.0 * H[k] for k in ks])
    x = W.f32_to_bf16_bits(rows)[None]
    codes, _, s, _, _ = gpu_compress(x, block, tb.VARIANT_STATIC, entry=MMA)
    for i, k in enumerate(ks + ks):
        want = 0x7E if i < len(ks) else 0xFE
        assert codes[0, i, k] == want
        assert np.all(np.delete(codes[0, i], k) & 0x7F == 0)
    assert np.all(s == np.float32(np.sqrt(block * E_STAR) / 448.0))


def test_mma_sixteen_shards():
    rng = np.random.default_rng(44)
    x = W.f32_to_bf16_bits(rng.normal(0, 1.0, size=(16, 9, 256)).astype(np.float32))
    check_compress_against_oracle(x, 128, entry=MMA)


@pytest.mark.parametrize("P,N,h,block", [(16, 2048, 1024, 64), (3, 40 * 128 // 16, 1024, 64), (5, 20000, 768, 256)])
def test_mma_tile_schedule(P, N, h, block, oracle_rows):
    """Shapes that drive the tile schedule through its cases: 16 shards (a few
    CTAs per shard, a claimed pool of about a quarter of the tiles), one tile
    per CTA (empty pool) and a ragged last tile in the pool. Every element
    against the CUDA-core compress and against the oracle; a second
    call on the same workspace gives the same codes, scales and headers."""
    rng = np.random.default_rng(P * 1000 + N)
    v = rng.laplace(0, 0.05, size=(P, N, h)).astype(np.float32)
    v[:, ::7, 3] *= 200.0
    x = W.f32_to_bf16_bits(v)
    ws = tb.new_workspace(P)
    xd = dev_bf16(x)
    b1, h1 = MMA(xd, block, workspace=ws)
    b2, h2 = MMA(xd, block, workspace=ws)
    torch.cuda.synchronize()
    assert GP.same_outputs(b1, h1, b2, h2, P, N, h, block)
    assert int(ws.count_nonzero()) == 0
    codes, alpha, s_, hdr, _ = gpu_compress(x, block, entry=MMA)
    fc, fa, fs, _, _ = gpu_compress(x, block)
    oc, oa, os_ = oracle_rows.compress(x, block, E_STAR)
    for p in range(P):
        parity.compare_codes(codes[p], fc[p], f"codes[{p}] vs CUDA-core path")
        parity.compare_scales(alpha[p], fa[p], f"alpha[{p}] vs CUDA-core path")
        parity.compare_scales(s_[p], fs[p], f"s[{p}] vs CUDA-core path")
        parity.compare_codes(codes[p], oc[p], f"codes[{p}] vs oracle")
        parity.compare_scales(alpha[p], oa[p], f"alpha[{p}] vs oracle")
        parity.compare_scales(s_[p], os_[p], f"s[{p}] vs oracle")
        assert hdr[p]["s_max"] == s_[p].max()
        assert hdr[p]["n_clamped"] == np.count_nonzero(s_[p] > 1.0)


def test_mma_empty_tensor():
    x = torch.empty((3, 0, 128), dtype=torch.bfloat16, device="cuda")
    _, headers = MMA(x, 64)
    hdr = tb.parse_headers(headers)
    assert list(hdr["s_max"]) == [0.0] * 3 and list(hdr["N"]) == [0] * 3


def test_mma_does_not_write_outside_its_buffers():
    w = W.WORKLOADS["gpt3-6.7b-grad"]
    N = 33
    x = dev_bf16(W.make_shards(w, N=N, P=2))
    sb = tb.shard_bytes(N, w.h, w.block)
    guard = 4096
    big = torch.full((2 * sb + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    bundle = big[guard: guard + 2 * sb].view(2, sb)
    MMA(x, w.block, bundle=bundle)
    torch.cuda.synchronize()
    assert bool((big[:guard] == 0xA5).all()) and bool((big[-guard:] == 0xA5).all())


def test_mma_deterministic_and_workspace_reset():
    w = W.WORKLOADS["gpt2-1.5b-act"]
    x = dev_bf16(W.make_shards(w, N=700, P=2))
    ws = tb.new_workspace(2)
    b1, h1 = MMA(x, w.block, workspace=ws)
    b2, h2 = MMA(x, w.block, workspace=ws)
    torch.cuda.synchronize()
    assert GP.same_outputs(b1, h1, b2, h2, 2, 700, w.h, w.block)
    assert int(ws.count_nonzero()) == 0      # counters and running totals


@pytest.mark.parametrize("entry", ["mma", "fwht", "recompress"])
def test_header_totals_over_the_full_grid(entry):
    """Per-tensor header from the running totals at full grid size: about
    one block in eight clamped (E* = 30000 puts the rotated rms at 173 code
    units) across every CTA, and the largest s in one constant block per
    shard (all its energy in one rotated coefficient); repeated calls give
    the same header and leave the workspace zero."""
    w = W.WORKLOADS["gpt2-1.5b-act"]
    E = 30000.0
    v = W.make_shards(w, P=2)
    one = W.f32_to_bf16_bits(np.array([0.5], np.float32))[0]
    v[0, -3, 128:192] = one
    v[1, w.N // 2 + 7, 0:64] = one ^ 0x8000
    x = dev_bf16(v)
    ws = tb.new_workspace(2)
    if entry == "recompress":
        bundle, _ = MMA(x, w.block, E)
        out = [tb.taco_reduce_recompress(bundle, 2, w.N, w.h, w.block, E, workspace=ws) for _ in range(2)]
        shards = [o[0][None] for o in out]
        headers = [o[1][None] for o in out]
        P = 1
    else:
        fn = MMA if entry == "mma" else tb.taco_compress_shards_fwht
        out = [fn(x, w.block, E, workspace=ws) for _ in range(2)]
        shards = [o[0] for o in out]
        headers = [o[1] for o in out]
        P = 2
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    assert torch.equal(headers[0], headers[1])
    _, _, s = tb.shard_views(shards[0], P, w.N, w.h, w.block)
    s = s.cpu().numpy()
    hdr = tb.parse_headers(headers[0])
    for p in range(P):
        assert np.count_nonzero(s[p] > 1.0) > 1000
        assert hdr[p]["s_max"] == s[p].max() and hdr[p]["s_max"] > 2.0
        assert hdr[p]["n_clamped"] == np.count_nonzero(s[p] > 1.0)


@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX])
def test_headers_per_shard_under_the_shared_tile_pool(variant, oracle_rows):
    """Eight shards, about a quarter of whose tiles go to one pool that every
    CTA claims from, shards interleaved, so a CTA compresses tiles of other
    shards than its own. Every header must still reduce its own shard's s
    only: each shard has its own seeded data (so its own largest s and its
    own count of s > 1; E* = 30000 clamps about one block in eight under
    DUAL), and the headers are compared with the oracle's s of that shard.
    A tile folded into another shard's totals moves a count or a maximum."""
    P, N, h, n, E = 8, 2048, 1600, 64, 30000.0
    x = W.make_shards(W.WORKLOADS["gpt2-1.5b-act"], N=N, P=P)
    ws = tb.new_workspace(P)
    bundle, headers = MMA(dev_bf16(x), n, E, variant, workspace=ws)
    codes, alpha, s = tb.shard_views(bundle, P, N, h, n)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    codes, alpha, s = codes.cpu().numpy(), alpha.cpu().numpy(), s.cpu().numpy()
    hdr = tb.parse_headers(headers)
    oc, oa, os_ = oracle_rows.compress(x, n, E, variant)
    maxima = set()
    for p in range(P):
        parity.compare_codes(codes[p], oc[p], f"codes[{p}]")
        parity.compare_scales(alpha[p], oa[p], f"alpha[{p}]")
        parity.compare_scales(s[p], os_[p], f"s[{p}]")
        assert hdr[p]["s_max"] == s[p].max()
        assert abs(hdr[p]["s_max"] - os_[p].max()) <= 1e-6 * os_[p].max()
        assert hdr[p]["n_clamped"] == np.count_nonzero(s[p] > 1.0)
        near_one = np.count_nonzero(np.abs(os_[p].astype(np.float64) - 1.0) < 1e-6)
        assert abs(int(hdr[p]["n_clamped"]) - np.count_nonzero(os_[p] > 1.0)) <= near_one
        maxima.add(float(hdr[p]["s_max"]))
    assert len(maxima) == P                  # the shards' headers differ
    if variant == tb.VARIANT_DUAL:
        assert min(int(hdr[p]["n_clamped"]) for p in range(P)) > 100


FULL = ["tiny-512x1024", "gpt2-1.5b-act", "gpt3-6.7b-act", "gpt3-6.7b-grad", "qwen-7b-long"]


@pytest.mark.parametrize("name", FULL)
def test_mma_full_size_every_element_and_against_cuda_core_path(name, oracle_rows):
    """The benchmark's compress launch at full size: every code, alpha and s
    against the oracle and against the CUDA-core compress (same parity bar),
    header as the reduction of s."""
    from oracle_rows import cached_compress
    w = W.WORKLOADS[name]
    x = W.make_shards(w)
    codes, alpha, s, hdr, _ = gpu_compress(x, w.block, entry=MMA)
    oc, oa, os_ = cached_compress(oracle_rows, name, x, w.block, E_STAR)
    stats = []
    for p in range(w.P):
        stats.append(parity.compare_codes(codes[p], oc[p], f"{name} codes[{p}]"))
        parity.compare_scales(alpha[p], oa[p], f"{name} alpha[{p}]")
        parity.compare_scales(s[p], os_[p], f"{name} s[{p}]")
        assert hdr[p]["s_max"] == s[p].max()
        assert hdr[p]["n_clamped"] == np.count_nonzero(s[p] > 1.0)
    report(f"{name} tensor-core compress", stats)
    fc, fa, fs, _, _ = gpu_compress(x, w.block)
    for p in range(w.P):
        parity.compare_codes(codes[p], fc[p], f"{name} codes[{p}] vs CUDA-core path")
        parity.compare_scales(alpha[p], fa[p], f"{name} alpha[{p}] vs CUDA-core path")
        parity.compare_scales(s[p], fs[p], f"{name} s[{p}] vs CUDA-core path")


def test_mma_no_wait_timed_out():
    """No bounded wait of the tensor-core kernel gave up in the cases above."""
    assert tb.taco_get_fault() & 8 == 0

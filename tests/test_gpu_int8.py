"""INT8 fallback format (taco_compress_shards_int8 / taco_decompress_reduce_int8)
against the CPU oracle run with the INT8 code format.

Bar: codes at least 99.99% equal and otherwise one integer apart, alpha and
s within 1e-6 relative, reconstructions within 1e-3 relative RMS; -128 is
never written.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O
from test_gpu_parity import E_STAR, bundle_from_arrays, dev_bf16, gpu_compress, host_bits

pytestmark = pytest.mark.gpu

I8 = O.FORMAT_INT8


def check_int8_against_oracle(x_bits, block, variant=tb.VARIANT_DUAL, target=E_STAR):
    codes, alpha, s, hdr, bundle = gpu_compress(x_bits, block, variant, target, tb.taco_compress_shards_int8)
    for p in range(x_bits.shape[0]):
        oc, oa, os_, oh = O.compress(x_bits[p], block, target, variant, I8)
        parity.compare_int8_codes(codes[p], oc, f"int8 codes[{p}]")
        parity.compare_scales(alpha[p], oa, f"alpha[{p}]")
        parity.compare_scales(s[p], os_, f"s[{p}]")
        assert hdr[p]["q_max"] == 127.0 and hdr[p]["variant"] == variant
        assert abs(hdr[p]["s_max"] - oh["s_max"]) <= 1e-6 * max(oh["s_max"], 1.0)
        near_one = np.count_nonzero(np.abs(os_.astype(np.float64) - 1.0) < 1e-6)
        assert abs(int(hdr[p]["n_clamped"]) - oh["n_clamped"]) <= near_one
    assert not np.any(codes == 0x80)
    return codes, alpha, s, bundle


@pytest.mark.parametrize("name,rows", [("tiny-512x1024", 96), ("gpt2-1.5b-act", 37),
                                       ("gpt3-6.7b-act", 29), ("gpt3-6.7b-grad", 23)])
def test_int8_compress_small(name, rows):
    w = W.WORKLOADS[name]
    check_int8_against_oracle(W.make_shards(w, N=rows, P=min(w.P, 3)), w.block)


@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX, tb.VARIANT_STATIC])
def test_int8_variants_and_targets(block, variant):
    rng = np.random.default_rng(block + 10 * variant + 7)
    v = rng.laplace(0, 0.02, size=(2, 41, 3 * block))
    v[:, :, 5] *= 300.0
    x = W.f32_to_bf16_bits(v.astype(np.float32))
    for target in (E_STAR, 900.0, 150.0):
        check_int8_against_oracle(x, block, variant, target)


@pytest.mark.parametrize("block", [64, 128, 256])
def test_int8_closed_forms(block):
    """Spike block -> every code +-64 (= sqrt(E*)), constant block -> one +-127; both
    reconstruct the input exactly."""
    H = O.sylvester_hadamard(block)
    rows = [np.zeros(block, np.float32) for _ in range(2)]
    rows[0][3] = -2.5
    rows.append(np.full(block, 0.0078125, np.float32))
    x = W.f32_to_bf16_bits(np.stack(rows))[None]
    codes, alpha, s, hdr, bundle = gpu_compress(x, block, entry=tb.taco_compress_shards_int8)
    q = codes.view(np.int8).astype(np.int64)
    assert np.array_equal(q[0, 0], np.where(-H[:, 3] > 0, 64, -64))
    assert np.all(q[0, 1] == 0) and alpha[0, 1, 0] == 1.0 and s[0, 1, 0] == 1.0
    assert q[0, 2, 0] == 127 and np.all(q[0, 2, 1:] == 0)
    out = tb.taco_decompress_reduce_int8(bundle, 1, 3, block, block)
    assert np.array_equal(host_bits(out), x[0])


@pytest.mark.parametrize("block,P", [(64, 4), (128, 8), (256, 3)])
def test_int8_decompress_from_oracle_codes(block, P):
    rng = np.random.default_rng(block * P)
    N, h = 29, 3 * block
    v = rng.laplace(0, 0.02, size=(P, N, h)).astype(np.float32)
    x = W.f32_to_bf16_bits(v)
    parts = [O.compress(x[p], block, 900.0, O.VARIANT_DUAL, I8) for p in range(P)]
    codes = np.stack([c for c, _, _, _ in parts])
    alpha = np.stack([a for _, a, _, _ in parts])
    s = np.stack([sc for _, _, sc, _ in parts])
    out = tb.taco_decompress_reduce_int8(bundle_from_arrays(codes, alpha, s, block), P, N, h, block)
    want = O.bf16_bits_to_f64(O.decompress_reduce(codes, alpha, s, block, I8))
    parity.compare_recon(O.bf16_bits_to_f64(host_bits(out)), want)


def test_int8_decode_every_byte():
    """Every signed byte value in every lane position: codes 0..255 in one block row."""
    block = 256
    codes = np.arange(256, dtype=np.uint8)[None, None, :]
    alpha = np.ones((1, 1, 1), np.float32)
    s = np.ones((1, 1, 1), np.float32)
    out = tb.taco_decompress_reduce_int8(bundle_from_arrays(codes, alpha, s, block), 1, 1, block, block)
    want = O.decompress_reduce(codes, alpha, s, block, I8)
    assert np.array_equal(host_bits(out), want)


def test_int8_empty_tensor():
    x = torch.empty((2, 0, 256), dtype=torch.bfloat16, device="cuda")
    _, headers = tb.taco_compress_shards_int8(x, 128)
    hdr = tb.parse_headers(headers)
    assert list(hdr["q_max"]) == [127.0, 127.0] and list(hdr["s_max"]) == [0.0, 0.0]


@pytest.mark.parametrize("name", ["gpt2-1.5b-act", "gpt3-6.7b-grad"])
def test_int8_full_size_every_element(name, oracle_rows):
    """Full size: every INT8 code, alpha and s against the oracle, and the
    GPU's compress + decompress-reduce against the oracle's, every element."""
    w = W.WORKLOADS[name]
    x = W.make_shards(w)
    codes, alpha, s, hdr, bundle = gpu_compress(x, w.block, entry=tb.taco_compress_shards_int8)
    oc, oa, os_ = oracle_rows.compress(x, w.block, E_STAR, O.VARIANT_DUAL, I8)
    for p in range(w.P):
        parity.compare_int8_codes(codes[p], oc[p], f"{name} codes[{p}]")
        parity.compare_scales(alpha[p], oa[p], f"{name} alpha[{p}]")
        parity.compare_scales(s[p], os_[p], f"{name} s[{p}]")
        assert hdr[p]["s_max"] == s[p].max()
    assert not np.any(codes == 0x80)
    out = host_bits(tb.taco_decompress_reduce_int8(bundle, w.P, w.N, w.h, w.block))
    want = oracle_rows.decompress_reduce(oc, oa, os_, w.block, I8)
    parity.compare_recon(O.bf16_bits_to_f64(out), O.bf16_bits_to_f64(want))


def _random_int8_bundle(N, h, block, P, seed):
    rng = np.random.default_rng(seed)
    K = h // block
    codes = np.clip(np.rint(rng.normal(0, 30, size=(P, N, h))), -127, 127).astype(np.int8).view(np.uint8)
    alpha = np.exp(rng.normal(np.log(3000.0), 0.5, size=(P, N, K))).astype(np.float32)
    s = np.where(rng.random((P, N, K)) < 0.9, 1.0, rng.uniform(1, 4, (P, N, K))).astype(np.float32)
    return codes, alpha, s


@pytest.mark.parametrize("block,P", [(64, 4), (128, 3), (256, 2)])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_STATIC])
def test_int8_reduce_recompress(block, P, variant):
    N, h = 21, 3 * block
    codes, alpha, s = _random_int8_bundle(N, h, block, P, seed=block * P + variant)
    bundle = bundle_from_arrays(codes, alpha, s, block)
    shard, header, _ = tb.taco_reduce_recompress_int8_ptrs([bundle[p] for p in range(P)], N, h, block,
                                                           900.0, variant)
    rc, ra, rs = tb.shard_views(shard.view(1, -1), 1, N, h, block)
    torch.cuda.synchronize()
    oc, oa, os_, oh = O.reduce_recompress(codes, alpha, s, block, 900.0, variant, I8)
    parity.compare_int8_codes(rc.cpu().numpy()[0], oc)
    parity.compare_scales(ra.cpu().numpy()[0], oa, "alpha")
    parity.compare_scales(rs.cpu().numpy()[0], os_, "s")
    assert tb.parse_headers(header.view(1, -1))[0]["q_max"] == 127.0


@pytest.mark.parametrize("block,P", [(64, 5), (128, 3), (256, 2)])
def test_int8_decompress_shards(block, P):
    N, h = 19, 3 * block
    codes, alpha, s = _random_int8_bundle(N, h, block, P, seed=block + P)
    bundle = bundle_from_arrays(codes, alpha, s, block)
    out = tb.taco_decompress_shards_int8_ptrs([bundle[p] for p in range(P)], N, h, block)
    for p in range(P):
        want = O.decompress_reduce(codes[p:p + 1], alpha[p:p + 1], s[p:p + 1], block, I8)
        parity.compare_recon(O.bf16_bits_to_f64(host_bits(out[p])), O.bf16_bits_to_f64(want))


def test_int8_no_wait_timed_out():
    assert tb.taco_get_fault() == 0

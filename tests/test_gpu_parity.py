"""CUDA path against the CPU oracle, through the C ABI (libtaco).

Small cases run the oracle on every element; full-size cases run the exact
launches the benchmark times and check every element against the oracle
(run unchanged over row ranges in worker processes), plus properties that
hold at any size.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import parity
from grads_taco_compress_gb300 import binding as tb
from grads_taco_compress_gb300 import workloads as W
from oracle import taco_oracle as O

pytestmark = pytest.mark.gpu

E_STAR = 4096.0


# ------------------------------------------------------------------ utils ----
def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bundle_from_arrays(codes, alpha, s, block) -> torch.Tensor:
    """Lay out (codes, alpha, s) [P,...] in the shard format, on the device."""
    P, N, h = codes.shape
    sb = tb.shard_bytes(N, h, block)
    off = tb.shard_scales_offset(N, h, block)
    buf = np.zeros((P, max(sb, 1)), dtype=np.uint8)
    for p in range(P):
        buf[p, : N * h] = codes[p].reshape(-1)
        pairs = np.stack([np.asarray(alpha[p], np.float32), np.asarray(s[p], np.float32)], axis=-1)
        buf[p, off: off + pairs.nbytes] = np.ascontiguousarray(pairs).view(np.uint8).reshape(-1)
    return torch.from_numpy(buf).cuda()


def gpu_compress(x_bits: np.ndarray, block: int, variant=tb.VARIANT_DUAL, target=E_STAR,
                 entry=tb.taco_compress_shards_fwht):
    """x_bits [P,N,h] -> (codes, alpha, s, headers) as numpy, via a compress entry."""
    P, N, h = x_bits.shape
    bundle, headers = entry(dev_bf16(x_bits), block, target, variant)
    codes, alpha, s = tb.shard_views(bundle, P, N, h, block)
    torch.cuda.synchronize()
    return (codes.cpu().numpy(), alpha.cpu().numpy(), s.cpu().numpy(),
            tb.parse_headers(headers), bundle)


def check_compress_against_oracle(x_bits, block, variant=tb.VARIANT_DUAL, target=E_STAR,
                                  entry=tb.taco_compress_shards_fwht):
    codes, alpha, s, hdr, _ = gpu_compress(x_bits, block, variant, target, entry)
    stats = []
    for p in range(x_bits.shape[0]):
        oc, oa, os_, oh = O.compress(x_bits[p], block, target, variant)
        stats.append(parity.compare_codes(codes[p], oc, f"codes[{p}]"))
        parity.compare_scales(alpha[p], oa, f"alpha[{p}]")
        parity.compare_scales(s[p], os_, f"s[{p}]")
        assert hdr[p]["N"] == x_bits.shape[1] and hdr[p]["h"] == x_bits.shape[2]
        assert hdr[p]["block"] == block and hdr[p]["variant"] == variant
        assert hdr[p]["q_max"] == 448.0 and hdr[p]["target_energy"] == np.float32(target)
        assert abs(hdr[p]["s_max"] - oh["s_max"]) <= 1e-6 * max(oh["s_max"], 1.0)
        # n_clamped may differ only where s sits within rounding of 1
        near_one = np.count_nonzero(np.abs(os_.astype(np.float64) - 1.0) < 1e-6)
        assert abs(int(hdr[p]["n_clamped"]) - oh["n_clamped"]) <= near_one
    return codes, alpha, s, hdr, stats


# ------------------------------------------------------------ E4M3 codec ----
def test_e4m3_encode_every_bf16_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32)
    v = (bits << 16).view(np.float32)
    got = tb.taco_e4m3_encode_f32(torch.from_numpy(v.copy()).cuda()).cpu().numpy()
    assert np.array_equal(got, O.e4m3_encode(v))


def test_e4m3_encode_ties_and_random_fp32():
    table = O.e4m3_decode_table()[:127]
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    rng = np.random.default_rng(21)
    rnd = (rng.standard_normal(1 << 20) * np.exp2(rng.uniform(-14, 10, 1 << 20))).astype(np.float32)
    v = np.concatenate([mids, -mids, rnd, np.float32([448, 464, 480, 1e30, -1e30, np.inf, -np.inf])])
    got = tb.taco_e4m3_encode_f32(torch.from_numpy(v).cuda()).cpu().numpy()
    assert np.array_equal(got, O.e4m3_encode(v))


def test_e4m3_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got = tb.taco_e4m3_decode_f32(torch.from_numpy(codes).cuda()).cpu().numpy().astype(np.float64)
    want = O.e4m3_decode_table()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


# ------------------------------------------------- compress, small cases ----
SMALL = [
    # (workload, rows): every config's value mix at a size the oracle checks
    # element by element; the row counts leave a ragged last warp tile.
    ("tiny-512x1024", 512),
    ("gpt2-1.5b-act", 37),
    ("gpt3-6.7b-act", 29),
    ("gpt3-6.7b-grad", 23),
    ("qwen-7b-long", 19),
]


@pytest.mark.parametrize("name,rows", SMALL)
def test_compress_small(name, rows):
    w = W.WORKLOADS[name]
    x = W.make_shards(w, N=rows, P=min(w.P, 3))
    _, _, _, _, stats = check_compress_against_oracle(x, w.block)
    assert all(s["equal_fraction"] >= parity.CODE_EQUAL_FRACTION for s in stats)


@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("variant", [tb.VARIANT_DUAL, tb.VARIANT_ABSMAX, tb.VARIANT_STATIC])
def test_compress_variants_and_targets(block, variant):
    rng = np.random.default_rng(block + 10 * variant)
    v = rng.laplace(0, 0.02, size=(2, 41, 3 * block))
    v[:, :, 5] *= 300.0                              # an outlier channel -> clamped blocks
    x = W.f32_to_bf16_bits(v.astype(np.float32))
    for target in (E_STAR, 1.0, 150.0):
        check_compress_against_oracle(x, block, variant, target)


@pytest.mark.parametrize("block", [64, 128, 256])
def test_compress_closed_form_blocks(block, entry=tb.taco_compress_shards_fwht):
    """Spike, constant and zero blocks: exact codes and exact round trip."""
    H = O.sylvester_hadamard(block)
    rows = []
    for j in (0, 7, block - 1):
        r = np.zeros(block, np.float32)
        r[j] = -2.5
        rows.append(r)
    rows.append(np.full(block, 0.0078125, np.float32))
    rows.append(np.zeros(block, np.float32))
    x = W.f32_to_bf16_bits(np.stack(rows))[None]
    codes, alpha, s, hdr, _ = gpu_compress(x, block, entry=entry)
    for i, j in enumerate((0, 7, block - 1)):
        want = np.where(-H[:, j] > 0, 0x68, 0xE8)
        assert np.array_equal(codes[0, i], want)
        assert s[0, i, 0] == 1.0
    assert codes[0, 3, 0] == 0x7E and np.all(codes[0, 3, 1:] & 0x7F == 0)
    assert abs(s[0, 3, 0] - np.sqrt(block * E_STAR) / 448.0) <= 2e-7 * s[0, 3, 0]
    assert np.all(codes[0, 4] & 0x7F == 0) and alpha[0, 4, 0] == 1.0 and s[0, 4, 0] == 1.0
    assert hdr[0]["n_clamped"] == 1
    out = tb.taco_decompress_reduce(bundle_from_arrays(codes, alpha, s, block), 1, 5, block, block)
    assert np.array_equal(host_bits(out), x[0])


def test_compress_single_equals_shards():
    w = W.WORKLOADS["gpt2-1.5b-act"]
    x = W.make_shards(w, N=64, P=3)
    bundle, headers = tb.taco_compress_shards(dev_bf16(x), w.block)
    sb = tb.shard_bytes(64, w.h, w.block)
    for p in range(3):
        shard, header = tb.taco_compress(dev_bf16(x[p]), w.block)
        assert same_outputs(shard[None, :sb], header, bundle[p:p + 1, :sb], headers[p], 1, 64, w.h, w.block)


def same_outputs(b1, h1, b2, h2, P, N, h, block):
    """Two compress results hold the same codes, scale pairs and headers, bit
    for bit. The bundle's alignment padding is never written, so it is not
    compared."""
    v1 = tb.shard_views(b1, P, N, h, block)
    v2 = tb.shard_views(b2, P, N, h, block)
    same = all(torch.equal(a.view(torch.uint8 if a.dtype == torch.uint8 else torch.int32),
                           b.view(torch.uint8 if b.dtype == torch.uint8 else torch.int32))
               for a, b in zip(v1, v2))
    return same and torch.equal(h1, h2)


BOTH = [tb.taco_compress_shards, tb.taco_compress_shards_fwht]   # tensor-core kernel, CUDA-core FWHT


@pytest.mark.parametrize("entry", BOTH)
def test_compress_deterministic_and_workspace_reset(entry):
    w = W.WORKLOADS["gpt3-6.7b-act"]
    x = dev_bf16(W.make_shards(w, N=300, P=2))
    ws = tb.new_workspace(2)
    b1, h1 = entry(x, w.block, workspace=ws)
    b2, h2 = entry(x, w.block, workspace=ws)
    torch.cuda.synchronize()
    assert same_outputs(b1, h1, b2, h2, 2, 300, w.h, w.block)
    assert int(ws.count_nonzero()) == 0      # counters and running totals


@pytest.mark.parametrize("entry", BOTH)
def test_compress_does_not_write_outside_its_buffers(entry):
    w = W.WORKLOADS["gpt3-6.7b-grad"]
    N = 33
    x = dev_bf16(W.make_shards(w, N=N, P=2))
    sb = tb.shard_bytes(N, w.h, w.block)
    guard = 4096
    big = torch.full((2 * sb + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    bundle = big[guard: guard + 2 * sb].view(2, sb)
    hbig = torch.full((2 * 40 + 2 * 64,), 0xA5, dtype=torch.uint8, device="cuda")
    headers = hbig[64: 64 + 80].view(2, 40)
    entry(x, w.block, bundle=bundle, headers=headers)
    torch.cuda.synchronize()
    assert bool((big[:guard] == 0xA5).all()) and bool((big[-guard:] == 0xA5).all())
    assert bool((hbig[:64] == 0xA5).all()) and bool((hbig[-64:] == 0xA5).all())


@pytest.mark.parametrize("entry", BOTH)
def test_compress_empty_tensor(entry):
    x = torch.empty((2, 0, 256), dtype=torch.bfloat16, device="cuda")
    bundle, headers = entry(x, 128)
    hdr = tb.parse_headers(headers)
    assert list(hdr["s_max"]) == [0.0, 0.0] and list(hdr["n_clamped"]) == [0, 0]
    assert list(hdr["N"]) == [0, 0]


def test_compress_one_block():
    x = W.f32_to_bf16_bits(np.linspace(-1, 1, 64, dtype=np.float32))[None, None]
    check_compress_against_oracle(x, 64)


def test_compress_wide_dynamic_range():
    """Magnitudes from 1e-12 to 1e12 inside one tensor (fp32 energy stays normal)."""
    rng = np.random.default_rng(31)
    mag = np.exp(rng.uniform(np.log(1e-12), np.log(1e12), size=(1, 17, 512)))
    v = mag * np.sign(rng.standard_normal((1, 17, 512)))
    v[:, ::3, :] = rng.normal(0, 1e-6, size=v[:, ::3, :].shape)   # quiet rows
    check_compress_against_oracle(W.f32_to_bf16_bits(v.astype(np.float32)), 128)


# --------------------------------------------- decompress-reduce, small ----
@pytest.mark.parametrize("name,rows", SMALL)
def test_decompress_reduce_small_from_oracle_codes(name, rows):
    w = W.WORKLOADS[name]
    x = W.make_shards(w, N=rows)
    parts = [O.compress(x[p], w.block, E_STAR) for p in range(w.P)]
    codes = np.stack([c for c, _, _, _ in parts])
    alpha = np.stack([a for _, a, _, _ in parts])
    s = np.stack([s_ for _, _, s_, _ in parts])
    out = tb.taco_decompress_reduce(bundle_from_arrays(codes, alpha, s, w.block), w.P, rows, w.h, w.block)
    got = O.bf16_bits_to_f64(host_bits(out))
    want_bits = O.decompress_reduce(codes, alpha, s, w.block)
    parity.compare_recon(got, O.bf16_bits_to_f64(want_bits))
    assert np.mean(host_bits(out) == want_bits) > 0.99


@pytest.mark.parametrize("block,P", [(64, 1), (64, 5), (128, 2), (128, 16), (256, 3), (256, 8)])
def test_decompress_reduce_random_bundles(block, P):
    N, h = 27, 3 * block
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=block + P)
    out = tb.taco_decompress_reduce(bundle_from_arrays(codes, alpha, s, block), P, N, h, block)
    want = O.bf16_bits_to_f64(O.decompress_reduce(codes, alpha, s, block))
    parity.compare_recon(O.bf16_bits_to_f64(host_bits(out)), want)


def test_decompress_reduce_ptrs_equals_bundle():
    block, P, N, h = 128, 4, 45, 512
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=3)
    bundle = bundle_from_arrays(codes, alpha, s, block)
    a = tb.taco_decompress_reduce(bundle, P, N, h, block)
    shards = [bundle[p].clone() for p in range(P)]
    b = tb.taco_decompress_reduce_ptrs(shards, N, h, block)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decompress_reduce_guards_and_empty():
    block, P, N, h = 64, 2, 19, 192
    codes, alpha, s = W.make_random_bundle(N, h, block, P, seed=4)
    bundle = bundle_from_arrays(codes, alpha, s, block)
    guard = 2048
    big = torch.full((N * h + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = big[guard: guard + N * h].view(N, h)
    tb.taco_decompress_reduce(bundle, P, N, h, block, out=out)
    torch.cuda.synchronize()
    assert bool((big[:guard] == -7.0).all()) and bool((big[-guard:] == -7.0).all())
    # N == 0: nothing is launched, nothing is written
    empty = torch.empty((0, h), dtype=torch.bfloat16, device="cuda")
    tb.taco_decompress_reduce(bundle, P, 0, h, block, out=empty)


def test_round_trip_through_gpu_is_close():
    w = W.WORKLOADS["tiny-512x1024"]
    x = W.make_shards(w)
    _, _, _, _, bundle = gpu_compress(x, w.block)
    out = tb.taco_decompress_reduce(bundle, w.P, w.N, w.h, w.block)
    ref = O.bf16_bits_to_f64(x).sum(axis=0)
    assert parity.rel_rms(O.bf16_bits_to_f64(host_bits(out)), ref) < 0.05


# ------------------------------------------------- full sizes, every element ----
FULL = ["tiny-512x1024", "gpt2-1.5b-act", "gpt3-6.7b-act", "gpt3-6.7b-grad", "qwen-7b-long"]


def report(what: str, stats: list) -> None:
    """One line per config: the share of codes equal to the oracle's and the worst step."""
    eq = min(st["equal_fraction"] for st in stats)
    worst = max(st["max_steps"] for st in stats)
    print(f"\nPARITY {what}: codes equal {eq:.6%} (worst shard), max {worst} step(s)")


@pytest.mark.parametrize("name", FULL)
def test_full_size_compress_every_element(name, oracle_rows):
    """The CUDA-core compress launch (all P shards at once) at full size:
    every code, alpha and s against the oracle."""
    from oracle_rows import cached_compress
    w = W.WORKLOADS[name]
    x = W.make_shards(w)
    codes, alpha, s, hdr, _ = gpu_compress(x, w.block)
    oc, oa, os_ = cached_compress(oracle_rows, name, x, w.block, E_STAR)
    stats = []
    for p in range(w.P):
        stats.append(parity.compare_codes(codes[p], oc[p], f"{name} codes[{p}]"))
        parity.compare_scales(alpha[p], oa[p], f"{name} alpha[{p}]")
        parity.compare_scales(s[p], os_[p], f"{name} s[{p}]")
        # header = reduction of the whole s array
        assert hdr[p]["s_max"] == s[p].max()
        assert hdr[p]["n_clamped"] == np.count_nonzero(s[p] > 1.0)
    report(f"{name} CUDA-core compress", stats)


@pytest.mark.parametrize("name", FULL)
def test_full_size_decompress_reduce_every_element(name, oracle_rows):
    """The benchmark's decompress-reduce launch at full size on a generated
    bundle: every output element against the oracle."""
    w = W.WORKLOADS[name]
    codes, alpha, s = W.make_random_bundle(w.N, w.h, w.block, w.P, seed=5)
    out = tb.taco_decompress_reduce(bundle_from_arrays(codes, alpha, s, w.block), w.P, w.N, w.h, w.block)
    got = host_bits(out)
    want = oracle_rows.decompress_reduce(codes, alpha, s, w.block)
    r = parity.compare_recon(O.bf16_bits_to_f64(got), O.bf16_bits_to_f64(want))
    same = float(np.mean(got == want))
    print(f"\nPARITY {name} decompress-reduce (generated bundle): bf16 equal {same:.6%}, rel RMS {r:.2e}")
    assert same > 0.99


@pytest.mark.parametrize("name", FULL)
def test_full_size_pipeline_every_element(name, oracle_rows):
    """The benchmark's step end to end at full size: the GPU's tensor-core
    compress then its decompress-reduce, against the oracle's compress then
    the oracle's decompress-reduce of the same seeded input, every element."""
    from oracle_rows import cached_compress
    w = W.WORKLOADS[name]
    x = W.make_shards(w)
    bundle, _ = tb.taco_compress_shards_mma(dev_bf16(x), w.block)
    got = host_bits(tb.taco_decompress_reduce(bundle, w.P, w.N, w.h, w.block))
    oc, oa, os_ = cached_compress(oracle_rows, name, x, w.block, E_STAR)
    want = oracle_rows.decompress_reduce(oc, oa, os_, w.block)
    r = parity.compare_recon(O.bf16_bits_to_f64(got), O.bf16_bits_to_f64(want))
    same = float(np.mean(got == want))
    print(f"\nPARITY {name} compress + decompress-reduce: bf16 equal {same:.6%}, rel RMS {r:.2e}")
    assert same > 0.99


@pytest.mark.parametrize("name", [n for n in FULL if n != "tiny-512x1024"])
def test_full_size_decompress_reduce_every_element(name):
    """Every output element of the full-size decompress-reduce is written and
    equals the sum of the P shards expanded on their own (taco_decompress_shards),
    within the bf16 roundings of the expansions. On the large workloads the
    warps claim their CTA's tiles in order; a tile skipped or taken twice would
    show here, where sampled rows could miss it."""
    w = W.WORKLOADS[name]
    codes, alpha, s = W.make_random_bundle(w.N, w.h, w.block, w.P, seed=6)
    bundle = bundle_from_arrays(codes, alpha, s, w.block)
    out = torch.full((w.N, w.h), 0x7FC0, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    tb.taco_decompress_reduce(bundle, w.P, w.N, w.h, w.block, out=out)
    parts = tb.taco_decompress_shards(bundle, w.P, w.N, w.h, w.block).float()
    torch.cuda.synchronize()
    got = out.float()
    assert bool(torch.isfinite(got).all())
    want = parts.sum(dim=0)
    # the bf16 roundings of the P expansions and of the sum (half an ulp:
    # up to 2^-8 relative each, 8 significant bits), plus the fp32 rounding
    # of both sides' Hadamard sums, which is relative to the block's
    # magnitude, not to the element's; a tile skipped or taken twice is off
    # by the whole value
    mag = parts.abs().sum(dim=0)
    bound = mag * 2.0 ** -7 + mag.max() * 2.0 ** -14
    excess = ((got - want).abs() - bound).max().item()
    assert excess <= 0.0, f"worst excess over the bound {excess:.3e} (max magnitude {mag.max().item():.3e})"


def test_no_kernel_wait_timed_out():
    """After every launch above, no bounded wait of any kernel gave up."""
    assert tb.taco_get_fault() == 0
